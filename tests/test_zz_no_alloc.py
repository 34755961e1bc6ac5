"""sp_attn_bwd_noalloc: the backward for callers that cannot allocate device memory
(code running where a framework owns all device memory, or under a fixed memory
plan).  It must give the results of sp_attn_bwd, whose workspace the caller
allocates, on consecutive calls that reuse the library's one scratch array.

This file is collected last so that a run stopping at its first failure has already
run every other test.
"""
import ctypes

import pytest
import torch

import oracle
from gpu_util import check_grad, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import binding, sp_attn_bwd, sp_attn_fwd, workloads

WORKSPACE = 6          # SP_ERR_WORKSPACE


def _inputs(B, H, sq, sk, d, seed):
    r = lambda shape, s: workloads.randn_bf16(shape, s, 1.0, device="cuda")
    return (r((B, sq, H, d), seed), r((B, sk, H, d), seed + 1), r((B, sk, H, d), seed + 2),
            r((B, sq, H, d), seed + 3))


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,sq,sk,d,causal,key_len", [
    (2, 3, 700, 700, 128, True, None),
    (3, 2, 300, 450, 64, False, [450, 200, 1]),
])
def test_noalloc_matches_workspace_backward_twice(B, H, sq, sk, d, causal, key_len):
    need_gpu()
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device="cuda")
    q, k, v, do = _inputs(B, H, sq, sk, d, 7 * sq + d)
    o, lse = sp_attn_fwd(q, k, v, causal, 0, kl)
    ref = sp_attn_bwd(q, k, v, o, lse, do, causal, 0, kl)
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()
    want = orc.attn_bwd(f64(q), f64(k), f64(v), f64(do), causal, 0, key_len)
    # two calls in a row: the second one finds the first one's leftovers in the scratch
    for call in range(2):
        got = binding.sp_attn_bwd_noalloc(q, k, v, o, lse, do, causal, 0, kl)
        torch.cuda.synchronize()
        check_status()
        # the same kernels run in the same order on the same inputs: dK and dV come out
        # of per-CTA accumulators and must be identical bit for bit; dQ is a sum of
        # atomically added fp32 pieces whose order may differ from run to run
        for name, a, b in zip(("dk", "dv"), got[1:], ref[1:]):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), \
                f"call {call} {name} differs from sp_attn_bwd"
        check_grad(f64(got[0]), f64(ref[0]), f"call {call} dq vs sp_attn_bwd")
        for name, a, r in zip(("dq", "dk", "dv"), got, want):
            check_grad(f64(a), r, f"call {call} {name} vs oracle")


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_the_scratch():
    """Needs more than SP_NOALLOC_SCRATCH_BYTES: refused before anything is launched
    (fake, never-dereferenced pointers are enough)."""
    lib = binding.load()
    p = binding.SpAttnParams()
    fake = 0x10000
    p.q = p.k = p.v = fake
    for name in ("q_stride", "k_stride", "v_stride", "o_stride"):
        setattr(p, name, (ctypes.c_int64 * 3)(64 * 4096 * 128, 64 * 128, 128))
    p.B, p.H, p.sq, p.sk, p.d = 1, 64, 4096, 4096, 128
    p.causal, p.q_offset, p.key_len, p.softmax_scale = 1, 0, None, 0.0
    assert lib.sp_attn_bwd_workspace_size(ctypes.byref(p)) > binding.NOALLOC_SCRATCH_BYTES
    assert lib.sp_attn_bwd_noalloc(ctypes.byref(p), fake, fake, fake, fake, fake, fake,
                                   None) == WORKSPACE
