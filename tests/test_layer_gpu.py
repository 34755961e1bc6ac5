"""The projections around attention on the GPU ("Parallel multi-head attention",
sections 2-3: ColumnParallel q/k/v projections, RowParallel output projection) and the
whole attention layer of the sequence-parallel step, against the fp64 oracle.

Bars: the projections and the layer round to bf16 several times in series (the packed
qkv, O, the output; each at most 2^-9 relative), so outputs and gradients are compared by
relative Frobenius error <= 2e-2, the bar the attention gradients use."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import (AttentionLayer, sp_linear_bwd, sp_linear_fwd,
                                              workloads)

pytestmark = pytest.mark.gpu


def _randn(shape, seed, scale=1.0):
    return workloads.randn_bf16(shape, seed, scale, device="cuda")


@pytest.mark.parametrize("M,n_in,n_out", [(300, 256, 384), (1000, 128, 64), (8, 64, 1024)])
def test_linear_matches_oracle(M, n_in, n_out):
    need_gpu()
    x = _randn((M, n_in), M + 1)
    w = _randn((n_out, n_in), M + 2, n_in ** -0.5)
    dy = _randn((M, n_out), M + 3)
    y = sp_linear_fwd(x, w)
    dx, dw = sp_linear_bwd(dy, x, w)
    dw2 = dw.clone()
    sp_linear_bwd(dy, x, w, dx=None, dw=dw2, accumulate_dw=True, need_dx=False)
    torch.cuda.synchronize()
    check_status()
    ry = oracle.linear_fwd(f64(x), f64(w))
    rdx, rdw = oracle.linear_bwd(f64(dy), f64(x), f64(w))
    check_grad(f64(y), ry, "y")
    check_grad(f64(dx), rdx, "dx")
    check_grad(f64(dw), rdw, "dw")
    check_grad(f64(dw2), 2 * rdw, "dw accumulated twice")


def _check_rounded(got: np.ndarray, ref: np.ndarray, what: str, roundings: int = 1):
    """Element by element: the inputs are bf16 values (exact in fp64), so the only errors
    are the fp32 accumulation order (far below bf16's precision) and the rounding of the
    result to bf16 (at most 2^-9 relative, once per rounding)."""
    bound = roundings * 2.0 ** -8 * np.abs(ref) + 1e-5 * max(np.abs(ref).max(), 1e-30)
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{what}: {bad.sum()} elements off, worst at "
                           f"{np.unravel_index(np.argmax(np.abs(got - ref) - bound), ref.shape)}")


@pytest.mark.parametrize("M,n_in,n_out", [
    (4100, 520, 776),      # every dimension ragged against the 128 x 256 x 64 tiles
    (8192, 1024, 2048),    # several tiles per persistent CTA in all three products
    (200, 24, 40),         # k shorter than one 64-wide stage
    (129, 8, 8),           # the smallest row width
    (1, 72, 264),          # one row: dW contracts over a single row, one ragged tile each
])
def test_linear_elementwise(M, n_in, n_out):
    """The tcgen05 GEMM behind the projections, every output element against the fp64
    oracle: y = x W^T (both operands k-contiguous), dx = dy W (W read n-contiguous) and
    dW (+)= dy^T x (both operands read m/n-contiguous)."""
    need_gpu()
    x = _randn((M, n_in), 7 * M + 1)
    w = _randn((n_out, n_in), 7 * M + 2, n_in ** -0.5)
    dy = _randn((M, n_out), 7 * M + 3)
    y = sp_linear_fwd(x, w)
    dx, dw = sp_linear_bwd(dy, x, w)
    dw2 = dw.clone()
    sp_linear_bwd(dy, x, w, dx=None, dw=dw2, accumulate_dw=True, need_dx=False)
    torch.cuda.synchronize()
    check_status()
    ry = oracle.linear_fwd(f64(x), f64(w))
    rdx, rdw = oracle.linear_bwd(f64(dy), f64(x), f64(w))
    _check_rounded(f64(y), ry, "y")
    _check_rounded(f64(dx), rdx, "dx")
    _check_rounded(f64(dw), rdw, "dw")
    _check_rounded(f64(dw2), 2 * rdw, "dw accumulated twice", roundings=2)


def test_linear_zero_rows():
    """M = 0: y and dx have no elements, dW = dy^T x is the zero matrix (cleared over an
    uninitialised buffer), and a dW accumulated into keeps its value."""
    need_gpu()
    w = _randn((40, 72), 5)
    x = torch.empty((0, 72), dtype=torch.bfloat16, device="cuda")
    dy = torch.empty((0, 40), dtype=torch.bfloat16, device="cuda")
    assert sp_linear_fwd(x, w).shape == (0, 40)
    dw = torch.full_like(w, 3.0)
    dx, dw = sp_linear_bwd(dy, x, w, dw=dw)
    kept = sp_linear_bwd(dy, x, w, dw=torch.full_like(w, 3.0), accumulate_dw=True)[1]
    torch.cuda.synchronize()
    check_status()
    assert dx.shape == (0, 72) and torch.count_nonzero(dw) == 0
    assert bool((kept == 3.0).all())


@pytest.mark.parametrize("N,b,s,h,d,dim", [(2, 1, 512, 4, 64, 256), (4, 2, 1024, 8, 128, 512)])
def test_layer_matches_oracle(N, b, s, h, d, dim):
    need_gpu()
    x = _randn((N, b, s // N, dim), 40 + s)
    wqkv = _randn((3 * h * d, dim), 41 + s, dim ** -0.5)
    wo = _randn((dim, h * d), 42 + s, (h * d) ** -0.5)
    dout = _randn((N, b, s // N, dim), 43 + s)
    layer = AttentionLayer(N, b, s, h, d, dim, causal=True)
    out = layer.forward(x, wqkv, wo)
    dx, dwqkv, dwo = layer.backward(dout)
    torch.cuda.synchronize()
    check_status()
    ref = oracle.Layer(oracle.default(), N, h, d, causal=True)
    rout = ref.forward(f64(x), f64(wqkv), f64(wo))
    rdx, rdwqkv, rdwo = ref.backward(f64(dout))
    check_grad(f64(out), rout, "layer out")
    check_grad(f64(dx), rdx, "layer dx")
    check_grad(f64(dwqkv), rdwqkv, "layer dwqkv")
    check_grad(f64(dwo), rdwo, "layer dwo")
