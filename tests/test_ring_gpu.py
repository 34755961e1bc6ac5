"""Ring / blockwise attention on the GPU ("adv07: Sequence Parallel", sections 5 and 7):
keys visited chunk by chunk (sp_attn_fwd with kv_offset, merged by sp_attn_merge), and
the backward chunk by chunk with the dQ accumulation.  Compared with the fp64 oracle's
attention over all keys (the split-key identity the oracle is pinned to), and the merge
step alone with the oracle's merge on the same partial results."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_lse, check_out, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import (ring_attention_bwd, ring_attention_fwd,
                                              sp_attn_fwd, sp_attn_merge, workloads)

pytestmark = pytest.mark.gpu


def _randn(shape, seed, scale=1.0):
    return workloads.randn_bf16(shape, seed, scale, device="cuda")


CASES = [
    # B, H, sq, sk, d, causal, q_offset, key_len, chunks (ragged, not tile aligned)
    (2, 3, 300, 700, 128, True, 400, None, [(0, 256), (256, 500), (500, 700)]),
    (2, 2, 333, 700, 64, False, 0, [700, 333], [(0, 128), (128, 300), (300, 700)]),
    (1, 2, 256, 256, 128, True, 0, None, [(0, 100), (100, 129), (129, 256)]),
    (1, 1, 130, 900, 128, True, 770, None, [(0, 300), (300, 600), (600, 900)]),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c[:7]) for c in CASES])
def test_ring_matches_full_attention(case):
    need_gpu()
    B, H, sq, sk, d, causal, q_offset, key_len, chunks = case
    seed = 31 * sq + sk
    q = _randn((B, sq, H, d), seed)
    k, v = _randn((B, sk, H, d), seed + 1), _randn((B, sk, H, d), seed + 2)
    do = _randn((B, sq, H, d), seed + 3)
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device="cuda")
    out, lse, _ = ring_attention_fwd(q, k, v, chunks, causal, q_offset, kl)
    dq, dk, dv = ring_attention_bwd(q, k, v, out, lse, do, chunks, causal, q_offset, kl)
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()
    ro, rl = orc.attn_fwd(f64(q), f64(k), f64(v), causal, q_offset, key_len)
    rdq, rdk, rdv = orc.attn_bwd(f64(q), f64(k), f64(v), f64(do), causal, q_offset, key_len)
    check_out(f64(out), ro, "ring out")
    check_lse(f64(lse), rl, "ring lse")
    check_grad(f64(dq), rdq, "ring dq (accumulated over chunks)")
    check_grad(f64(dk), rdk, "ring dk")
    check_grad(f64(dv), rdv, "ring dv")


def test_merge_matches_oracle_merge():
    """The merge kernel alone: the GPU's per-chunk partials merged on the GPU (fp32)
    against the same partials merged by the oracle (fp64)."""
    need_gpu()
    B, H, sq, sk, d = 2, 2, 200, 520, 128
    q = _randn((B, sq, H, d), 11)
    k, v = _randn((B, sk, H, d), 12), _randn((B, sk, H, d), 13)
    chunks = [(0, 200), (200, 390), (390, 520)]
    parts, lses = [], []
    o_acc = torch.empty((B, sq, H, d), dtype=torch.float32, device="cuda")
    lse_acc = torch.empty((B, H, sq), dtype=torch.float32, device="cuda")
    out = torch.empty_like(q)
    for n, (lo, hi) in enumerate(chunks):
        o, l = sp_attn_fwd(q, k[:, lo:hi], v[:, lo:hi], True, 300, kv_offset=lo)
        parts.append(o.clone())
        lses.append(l.clone())
        sp_attn_merge(o, l, o_acc, lse_acc, init=(n == 0), o_out=out if n == 2 else None)
    torch.cuda.synchronize()
    check_status()
    ro, rl = oracle.default().attn_merge([f64(p) for p in parts], [f64(l) for l in lses])
    assert np.abs(f64(o_acc) - ro).max() <= 1e-5
    fin = np.isfinite(rl)
    assert np.array_equal(np.isfinite(f64(lse_acc)), fin)
    assert np.abs(f64(lse_acc)[fin] - rl[fin]).max() <= 1e-5
    # the bf16 output is the accumulator rounded to nearest
    assert torch.equal(out, o_acc.to(torch.bfloat16))


def test_single_chunk_is_plain_attention_bit_exact():
    """One chunk: the merge has weight exactly 1, so ring attention returns the forward's
    own bf16 output and lse unchanged."""
    need_gpu()
    q, k, v = (_randn((2, 300, 3, 128), 20 + t) for t in range(3))
    ref, ref_lse = sp_attn_fwd(q, k, v, True)
    out, lse, _ = ring_attention_fwd(q, k, v, [(0, 300)], True)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(lse, ref_lse)


def test_chunk_invisible_to_every_row():
    """A causal key chunk that starts after the last query sees nothing: out 0, lse -inf,
    and merging it leaves the accumulator unchanged."""
    need_gpu()
    q = _randn((1, 128, 2, 64), 30)
    k, v = _randn((1, 512, 2, 64), 31), _randn((1, 512, 2, 64), 32)
    o, l = sp_attn_fwd(q, k[:, 256:], v[:, 256:], True, 0, kv_offset=256)
    torch.cuda.synchronize()
    assert not o.any() and torch.all(l == -float("inf"))
    full, full_lse, acc = ring_attention_fwd(q, k, v, [(0, 256), (256, 512)], True)
    head, head_lse = sp_attn_fwd(q, k[:, :256], v[:, :256], True)
    torch.cuda.synchronize()
    assert torch.equal(full.view(torch.int16), head.view(torch.int16))
    assert torch.equal(full_lse, head_lse)
