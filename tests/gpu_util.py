"""Helpers shared by the GPU parity tests: running libsp through the binding,
widening bf16 results for the fp64 oracle, and the comparison bars.

Tolerances (bf16 inputs, fp32 accumulation, bf16 outputs):
  out : max |gpu - oracle| <= 1e-2 and mean |gpu - oracle| <= 1e-3
  lse : max |gpu - oracle| <= 1e-2 (natural log)
  dq/dk/dv : ||gpu - oracle||_F / ||oracle||_F <= 2e-2
  relayout : bit-exact
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-2
GRAD_REL_FRO = 2e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().to("cpu").view(torch.int16).numpy().view(np.uint16)


def check_status():
    from sequence_head_attention_seq_b300 import sp_get_device_status
    code = sp_get_device_status()
    assert code == 0, f"device status {code}"


def check_out(gpu: np.ndarray, ref: np.ndarray, what: str):
    err = np.abs(gpu - ref)
    assert err.max() <= OUT_MAX_ABS, f"{what}: max abs {err.max():.3e}"
    assert err.mean() <= OUT_MEAN_ABS, f"{what}: mean abs {err.mean():.3e}"


def check_lse(gpu: np.ndarray, ref: np.ndarray, what: str):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isfinite(gpu), fin), f"{what}: -inf pattern differs"
    if fin.any():
        err = np.abs(gpu[fin] - ref[fin]).max()
        assert err <= LSE_MAX_ABS, f"{what}: max abs {err:.3e}"
    assert np.all(gpu[~fin] == -np.inf), f"{what}: empty rows must be -inf"


def check_grad(gpu: np.ndarray, ref: np.ndarray, what: str):
    nref = np.linalg.norm(ref)
    ndiff = np.linalg.norm(gpu - ref)
    if nref == 0.0:
        assert ndiff == 0.0, f"{what}: expected exact zeros"
        return
    rel = ndiff / nref
    assert rel <= GRAD_REL_FRO, f"{what}: rel Frobenius {rel:.3e}"
