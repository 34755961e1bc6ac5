"""General key mask on the GPU (transformers PR 31525 collator: attention_mask =
input_ids != pad_token_id, pads anywhere), forward and backward against the fp64
oracle on the same seeded inputs, plus the special cases the mask must reduce to."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_lse, check_out, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import sp_attn_bwd, sp_attn_fwd, workloads

pytestmark = pytest.mark.gpu


def _randn(shape, seed):
    return workloads.randn_bf16(shape, seed, 1.0, device="cuda")


def _mask(B, sk, seed, keep=0.7):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.rand((B, sk), generator=g) < keep


def _run(q, k, v, do, causal, q_offset=0, key_len=None, mask=None):
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device="cuda")
    km = None if mask is None else mask.to("cuda")
    o, lse = sp_attn_fwd(q, k, v, causal, q_offset, kl, key_mask=km)
    dq, dk, dv = sp_attn_bwd(q, k, v, o, lse, do, causal, q_offset, kl, key_mask=km)
    torch.cuda.synchronize()
    check_status()
    return o, lse, dq, dk, dv


CASES = [
    # B, H, sq, sk, d, causal, q_offset, key_len
    (3, 2, 300, 300, 128, True, 0, None),
    (3, 2, 257, 450, 64, False, 0, None),
    (2, 3, 200, 333, 128, True, 133, [333, 200]),
    (2, 1, 130, 1000, 64, False, 0, [1000, 777]),
]


@pytest.mark.parametrize("case", CASES, ids=[str(c) for c in CASES])
def test_key_mask_against_oracle(case):
    need_gpu()
    B, H, sq, sk, d, causal, q_offset, key_len = case
    seed = 13 * sq + sk
    q = _randn((B, sq, H, d), seed)
    k, v = _randn((B, sk, H, d), seed + 1), _randn((B, sk, H, d), seed + 2)
    do = _randn((B, sq, H, d), seed + 3)
    mask = _mask(B, sk, seed)
    mask[1, :] = False                     # a batch entry with no key at all
    mask[0, 128:256] = False               # a whole key block masked in batch entry 0
    o, lse, dq, dk, dv = _run(q, k, v, do, causal, q_offset, key_len, mask)
    orc = oracle.default()
    m = mask.numpy()
    ro, rl = orc.attn_fwd(f64(q), f64(k), f64(v), causal, q_offset, key_len, key_mask=m)
    rdq, rdk, rdv = orc.attn_bwd(f64(q), f64(k), f64(v), f64(do), causal, q_offset, key_len,
                                 key_mask=m)
    check_out(f64(o), ro, "out")
    check_lse(f64(lse), rl, "lse")
    check_grad(f64(dq), rdq, "dq")
    check_grad(f64(dk), rdk, "dk")
    check_grad(f64(dv), rdv, "dv")
    assert not o[1].any() and not dq[1].any() and not dk[1].any() and not dv[1].any()
    assert not dk[0, 128:256].any() and not dv[0, 128:256].any()


def test_right_padding_mask_equals_key_len():
    """A mask that keeps the first n keys is key_len = n: the same forward, bit for bit."""
    need_gpu()
    B, H, sq, sk, d = 2, 2, 260, 520, 128
    q = _randn((B, sq, H, d), 70)
    k, v = _randn((B, sk, H, d), 71), _randn((B, sk, H, d), 72)
    do = _randn((B, sq, H, d), 73)
    key_len = [520, 301]
    mask = torch.arange(sk)[None, :] < torch.tensor(key_len)[:, None]
    for causal in (True, False):
        a = _run(q, k, v, do, causal, 0, None, mask)
        b = _run(q, k, v, do, causal, 0, key_len, None)
        assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
        assert torch.equal(a[1], b[1])
        for x, y, n in zip(a[2:], b[2:], ("dq", "dk", "dv")):
            check_grad(f64(x), f64(y), n)


def test_left_padding_mask_equals_truncated_keys():
    """Non-causal, a mask that drops the first n keys: attention on the other keys."""
    need_gpu()
    B, H, sq, sk, d, n = 2, 2, 200, 400, 64, 150
    q = _randn((B, sq, H, d), 80)
    k, v = _randn((B, sk, H, d), 81), _randn((B, sk, H, d), 82)
    do = _randn((B, sq, H, d), 83)
    mask = (torch.arange(sk)[None, :] >= n).repeat(B, 1)
    a = _run(q, k, v, do, False, 0, None, mask)
    b = _run(q, k[:, n:].contiguous(), v[:, n:].contiguous(), do, False)
    check_out(f64(a[0]), f64(b[0]), "out")
    check_lse(f64(a[1]), f64(b[1]), "lse")
    check_grad(f64(a[2]), f64(b[2]), "dq")
    check_grad(f64(a[3][:, n:]), f64(b[3]), "dk")
    assert not a[3][:, :n].any() and not a[4][:, :n].any()
