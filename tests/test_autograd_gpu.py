"""The autograd entry points on the GPU: gradients through torch.autograd equal the direct
library calls (same kernels, same order: out, dK and dV bit for bit; dQ, whose fp32
additions land in any order, within the gradient bar) and the oracle; the all-to-all's
gradient is the inverse regrouping, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_out, check_status, f64, need_gpu, u16
from sequence_head_attention_seq_b300 import (UlyssesAttention, attention, seq_all_to_all,
                                              sp_attn_bwd, sp_attn_fwd, sp_relayout,
                                              ulysses_attention, workloads)

pytestmark = pytest.mark.gpu


def _randn(shape, seed, scale=1.0):
    return workloads.randn_bf16(shape, seed, scale, device="cuda")


def _bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    a, b = a.detach().contiguous(), b.detach().contiguous()
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


CASES = [
    # B, H, sq, sk, d, causal, q_offset, key_len, masked
    (2, 3, 300, 300, 128, True, 0, None, False),
    (2, 2, 257, 400, 64, False, 0, [400, 133], True),
    (1, 2, 200, 456, 128, True, 256, None, False),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_attention_autograd(case):
    need_gpu()
    B, H, sq, sk, d, causal, q_offset, key_len, masked = case
    seed = 13 * sq + sk
    q = _randn((B, sq, H, d), seed).requires_grad_()
    k = _randn((B, sk, H, d), seed + 1).requires_grad_()
    v = _randn((B, sk, H, d), seed + 2).requires_grad_()
    do = _randn((B, sq, H, d), seed + 3)
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device="cuda")
    km = None
    if masked:
        g = torch.Generator(device="cpu")
        g.manual_seed(seed + 4)
        km = (torch.rand((B, sk), generator=g) < 0.7).to("cuda")
    out = attention(q, k, v, causal, q_offset, kl, key_mask=km)
    dq, dk, dv = torch.autograd.grad(out, (q, k, v), do)
    o_ref, lse_ref = sp_attn_fwd(q.detach(), k.detach(), v.detach(), causal, q_offset, kl,
                                 key_mask=km)
    dq_ref, dk_ref, dv_ref = sp_attn_bwd(q.detach(), k.detach(), v.detach(), o_ref, lse_ref,
                                         do, causal, q_offset, kl, key_mask=km)
    torch.cuda.synchronize()
    check_status()
    assert _bits_equal(out, o_ref)
    assert _bits_equal(dk, dk_ref) and _bits_equal(dv, dv_ref)
    check_grad(f64(dq), f64(dq_ref), "dq against the direct call")
    mask = None if km is None else km.cpu().numpy()
    orc = oracle.default()
    qa, ka, va = f64(q), f64(k), f64(v)
    ro, _ = orc.attn_fwd(qa, ka, va, causal, q_offset, key_len, key_mask=mask)
    rdq, rdk, rdv = orc.attn_bwd(qa, ka, va, f64(do), causal, q_offset, key_len, key_mask=mask)
    check_out(f64(out), ro, "out")
    check_grad(f64(dq), rdq, "dq")
    check_grad(f64(dk), rdk, "dk")
    check_grad(f64(dv), rdv, "dv")


SHARDS = [
    # N, b, s, h, d, causal, key_len range
    (2, 1, 512, 4, 64, True, None),
    (4, 2, 1024, 8, 128, True, None),
    (2, 2, 512, 4, 128, False, (200, 512)),
]


@pytest.mark.parametrize("case", SHARDS, ids=[str(c) for c in SHARDS])
def test_ulysses_attention_autograd(case):
    """ulysses_attention (explicit regroupings, and fused into the kernels' addressing)
    against the UlyssesAttention step's forward and backward calls."""
    need_gpu()
    N, b, s, h, d, causal, klr = case
    shape = (N, b, s // N, h, d)
    seed = 7 * s + h
    q, k, v, do = (_randn(shape, seed + t) for t in range(4))
    kl = None
    if klr is not None:
        kl = workloads.key_lengths(b, klr[0], klr[1], seed + 5).to("cuda")
    step = UlyssesAttention(N, b, s, h, d, causal, key_len=kl)
    o_ref = step.forward(q, k, v).clone()
    dq_ref, dk_ref, dv_ref = (t.clone() for t in step.backward(do))
    for fused in (False, True):
        qq, kk, vv = (t.clone().requires_grad_() for t in (q, k, v))
        out = ulysses_attention(qq, kk, vv, causal, kl, fused=fused)
        dq, dk, dv = torch.autograd.grad(out, (qq, kk, vv), do)
        torch.cuda.synchronize()
        check_status()
        assert out.shape == shape
        assert _bits_equal(out, o_ref), f"out (fused={fused})"
        assert _bits_equal(dk, dk_ref) and _bits_equal(dv, dv_ref), f"dk/dv (fused={fused})"
        check_grad(f64(dq), f64(dq_ref), f"dq (fused={fused})")


def test_ulysses_attention_against_oracle():
    """One small step through autograd against the oracle's attention over the regrouped
    heads (the regrouping by the oracle's own index loop)."""
    need_gpu()
    N, b, s, h, d = 2, 1, 256, 4, 64
    shape = (N, b, s // N, h, d)
    q, k, v, do = (_randn(shape, 900 + t) for t in range(4))
    qq, kk, vv = (t.clone().requires_grad_() for t in (q, k, v))
    out = ulysses_attention(qq, kk, vv, True)
    dq, dk, dv = torch.autograd.grad(out, (qq, kk, vv), do)
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()

    def groups(t):   # shards -> [N*b][s][h/N][d] through the oracle's regrouping
        g = orc.seq2head(u16(t), N, b, s, h, d)
        return torch.from_numpy(g.view(np.int16)).view(torch.bfloat16).to(torch.float64) \
            .numpy().reshape(N * b, s, h // N, d)

    def shards(x):   # [N*b][s][h/N][d] -> [N][b][s/N][h][d]: shard r row u head g*h/N+j
        return x.reshape(N, b, N, s // N, h // N, d).transpose(2, 1, 3, 0, 4, 5).reshape(shape)

    qg, kg, vg, dog = groups(q), groups(k), groups(v), groups(do)
    ro, _ = orc.attn_fwd(qg, kg, vg, True)
    rdq, rdk, rdv = orc.attn_bwd(qg, kg, vg, dog, True)
    check_out(f64(out), shards(ro), "out")
    check_grad(f64(dq), shards(rdq), "dq")
    check_grad(f64(dk), shards(rdk), "dk")
    check_grad(f64(dv), shards(rdv), "dv")


def test_seq_all_to_all_gradient_is_the_inverse():
    need_gpu()
    N, b, s, h, d = 4, 2, 256, 8, 64
    x = _randn((N, b, s // N, h, d), 950).requires_grad_()
    y = seq_all_to_all(x, N, 2, 1)
    assert y.shape == (N, b, s, h // N, d)
    w = _randn(tuple(y.shape), 951)
    (gx,) = torch.autograd.grad(y, (x,), w)
    torch.cuda.synchronize()
    assert _bits_equal(y, sp_relayout(x.detach(), N, 2, 1))
    assert _bits_equal(gx, sp_relayout(w, N, 1, 2))
    back = seq_all_to_all(y, N, 1, 2)
    assert _bits_equal(back, x)
