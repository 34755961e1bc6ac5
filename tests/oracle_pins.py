"""Pins that tie the fp64 oracle to facts outside itself.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with something the pages or the mathematics fix:

* a library routine: torch's fp64 ``scaled_dot_product_attention`` and its
  autograd derivative, ``torch.logsumexp``, ``torch`` reshape/permute;
* closed forms: q = 0 (uniform weights), causal row 0, constant V, one key,
  two keys (a logistic weight);
* invariants: softmax rows sum to 1, column sums of dK vanish, column sums of
  dV equal those of dO, key padding equals truncation;
* central finite differences of sum(dO * out) for the backward;
* the pages' worked examples (fixtures under tests/golden/, each with its
  citation): the causal sequence-parallel example and the split-Q check of
  the "adv07: Sequence Parallel" tutorial, and hand-derived regrouping cases.

The same pins run against deliberately broken builds of the oracle (see
test_oracle_mutants.py) to show that each plausible mistake is caught.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _bhsd(x):
    """[B][S][H][d] numpy -> torch [B][H][S][d] fp64."""
    return torch.tensor(x, dtype=torch.float64).permute(0, 2, 1, 3).contiguous()


def _allowed(B, sq, sk, causal, q_offset, key_len, key_mask=None):
    """Boolean [B][1][sq][sk]: True where key j takes part for row i."""
    i = torch.arange(sq).view(sq, 1)
    j = torch.arange(sk).view(1, sk)
    m = torch.ones(B, 1, sq, sk, dtype=torch.bool)
    if causal:
        m &= (j <= i + q_offset).view(1, 1, sq, sk)
    if key_len is not None:
        kl = torch.tensor(np.asarray(key_len), dtype=torch.int64).view(B, 1, 1, 1)
        m &= j.view(1, 1, 1, sk) < kl
    if key_mask is not None:
        m &= torch.tensor(np.asarray(key_mask) != 0).view(B, 1, 1, sk)
    return m


def _torch_reference(q, k, v, dout, causal, q_offset, key_len, scale, key_mask=None):
    """torch fp64: out, lse, dq, dk, dv through sdpa + autograd (rows with no key dropped)."""
    B, sq, H, d = q.shape
    sk = k.shape[1]
    tq, tk, tv = (_bhsd(a).requires_grad_() for a in (q, k, v))
    mask = _allowed(B, sq, sk, causal, q_offset, key_len, key_mask)
    out = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    out = torch.nan_to_num(out, nan=0.0)           # rows with no visible key
    scores = torch.matmul(tq, tk.transpose(-1, -2)) * scale
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    rows_ok = mask.any(-1, keepdim=True)        # [B][1][sq][1]
    out = torch.where(rows_ok, out, torch.zeros_like(out))
    out.backward(_bhsd(dout))
    back = lambda t: t.permute(0, 2, 1, 3).detach().numpy()
    return (back(out), lse.detach().numpy(), back(tq.grad), back(tk.grad), back(tv.grad),
            rows_ok[:, 0, :, 0].numpy())


def _close(a, b, tol, what):
    a = np.asarray(a)
    b = np.asarray(b)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs diff {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- library routines

def pin_sdpa_causal_square(orc):
    """Causal, sq == sk: torch's fp64 sdpa(is_causal) and its autograd gradients."""
    B, H, S, d = 2, 3, 37, 16
    q, k, v, do = (_rand((B, S, H, d), 10 + t) for t in range(4))
    scale = 1.0 / math.sqrt(d)
    out, lse = orc.attn_fwd(q, k, v, True)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, True)
    tq, tk, tv = (_bhsd(a).requires_grad_() for a in (q, k, v))
    ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale)
    ref.backward(_bhsd(do))
    back = lambda t: t.permute(0, 2, 1, 3).detach().numpy()
    _close(out, back(ref), 1e-12, "out vs sdpa(is_causal)")
    _close(dq, back(tq.grad), 1e-11, "dq vs autograd")
    _close(dk, back(tk.grad), 1e-11, "dk vs autograd")
    _close(dv, back(tv.grad), 1e-11, "dv vs autograd")
    i = torch.arange(S)
    mask = (i.view(S, 1) >= i.view(1, S))
    sc = torch.matmul(_bhsd(q), _bhsd(k).transpose(-1, -2)) * scale
    _close(lse, torch.logsumexp(sc.masked_fill(~mask, float("-inf")), -1).numpy(), 1e-12,
           "lse vs torch.logsumexp")


def pin_sdpa_masks(orc):
    """q_offset, sq != sk and right-padded keys: sdpa with an explicit boolean mask."""
    B, H, d = 3, 2, 8
    for (sq, sk, causal, q_offset, key_len) in [
        (20, 45, True, 25, None),
        (20, 45, True, 25, [45, 30, 26]),
        (33, 50, False, 0, [50, 17, 1]),
        (33, 33, True, 0, [33, 9, 20]),
    ]:
        q = _rand((B, sq, H, d), 20 + sq)
        k, v = _rand((B, sk, H, d), 21 + sk), _rand((B, sk, H, d), 22 + sk)
        do = _rand((B, sq, H, d), 23)
        scale = 0.3
        out, lse = orc.attn_fwd(q, k, v, causal, q_offset, key_len, scale)
        dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, q_offset, key_len, scale)
        r_out, r_lse, r_dq, r_dk, r_dv, ok = _torch_reference(q, k, v, do, causal, q_offset,
                                                              key_len, scale)
        tag = f"sq={sq} sk={sk} causal={causal} off={q_offset} kl={key_len}"
        _close(out, r_out, 1e-12, "out " + tag)
        _close(np.where(ok[:, None, :], lse, 0), np.where(ok[:, None, :], r_lse, 0), 1e-12,
               "lse " + tag)
        _close(dq, r_dq, 1e-11, "dq " + tag)
        _close(dk, r_dk, 1e-11, "dk " + tag)
        _close(dv, r_dv, 1e-11, "dv " + tag)


def pin_sdpa_key_mask(orc):
    """A general key mask (transformers PR 31525 collator: attention_mask = input_ids != pad,
    pads anywhere), alone and combined with causal, q_offset and key_len: torch fp64 sdpa
    with the same boolean mask, and its autograd gradients.  One batch entry masks every
    key (out 0, lse -inf, no gradient)."""
    B, H, d = 3, 2, 8
    rng = np.random.default_rng(190)
    for (sq, sk, causal, q_offset, key_len) in [(21, 37, True, 16, None),
                                                (30, 30, False, 0, None),
                                                (19, 44, True, 25, [44, 30, 20])]:
        mask = rng.random((B, sk)) < 0.7
        mask[1, :] = False                         # a batch entry with no key at all
        mask[0, 0] = True
        q = _rand((B, sq, H, d), 191 + sq)
        k, v = _rand((B, sk, H, d), 192 + sk), _rand((B, sk, H, d), 193 + sk)
        do = _rand((B, sq, H, d), 194)
        scale = 0.4
        out, lse = orc.attn_fwd(q, k, v, causal, q_offset, key_len, scale, key_mask=mask)
        dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, q_offset, key_len, scale, key_mask=mask)
        r_out, r_lse, r_dq, r_dk, r_dv, ok = _torch_reference(q, k, v, do, causal, q_offset,
                                                              key_len, scale, mask)
        tag = f"sq={sq} sk={sk} causal={causal} off={q_offset} kl={key_len}"
        _close(out, r_out, 1e-12, "out " + tag)
        _close(np.where(ok[:, None, :], lse, 0), np.where(ok[:, None, :], r_lse, 0), 1e-12,
               "lse " + tag)
        assert np.all(lse[1] == -np.inf) and not out[1].any() and not dq[1].any()
        _close(dq, r_dq, 1e-11, "dq " + tag)
        _close(dk, r_dk, 1e-11, "dk " + tag)
        _close(dv, r_dv, 1e-11, "dv " + tag)


def pin_key_mask_special_cases(orc):
    """A mask that keeps the first n keys is right padding (key_len = n); all ones is no
    mask; a mask that drops the first n keys of a non-causal problem is attention on the
    remaining keys only."""
    B, H, sq, sk, d = 2, 2, 13, 29, 8
    q = _rand((B, sq, H, d), 200)
    k, v = _rand((B, sk, H, d), 201), _rand((B, sk, H, d), 202)
    do = _rand((B, sq, H, d), 203)
    key_len = [29, 11]
    right = np.arange(sk)[None, :] < np.array(key_len)[:, None]
    for causal in (True, False):
        a = orc.attn_fwd(q, k, v, causal, 5, key_mask=right)
        b = orc.attn_fwd(q, k, v, causal, 5, key_len)
        assert all(np.array_equal(x, y) for x, y in zip(a, b)), "right padding"
        a = orc.attn_bwd(q, k, v, do, causal, 5, key_mask=right)
        b = orc.attn_bwd(q, k, v, do, causal, 5, key_len)
        assert all(np.array_equal(x, y) for x, y in zip(a, b)), "right padding bwd"
        a = orc.attn_fwd(q, k, v, causal, 5, key_mask=np.ones((B, sk)))
        b = orc.attn_fwd(q, k, v, causal, 5)
        assert all(np.array_equal(x, y) for x, y in zip(a, b)), "all-ones mask"
    n = 9
    left = np.arange(sk)[None, :].repeat(B, 0) >= n
    out, lse = orc.attn_fwd(q, k, v, False, key_mask=left)
    ref, ref_lse = orc.attn_fwd(q, k[:, n:], v[:, n:], False)
    _close(out, ref, 1e-14, "left padding out")
    _close(lse, ref_lse, 1e-14, "left padding lse")


# ---------------------------------------------------------------- finite differences

def pin_finite_differences(orc):
    """Backward = gradient of L = sum(dO * out), by central differences in fp64."""
    B, H, sq, sk, d = 2, 2, 9, 13, 8
    q_offset, key_len, scale = 3, [13, 7], 0.4
    q, do = _rand((B, sq, H, d), 31), _rand((B, sq, H, d), 32)
    k, v = _rand((B, sk, H, d), 33), _rand((B, sk, H, d), 34)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, True, q_offset, key_len, scale)

    def loss(qq, kk, vv):
        out, _ = orc.attn_fwd(qq, kk, vv, True, q_offset, key_len, scale)
        return float(np.sum(out * do))

    rng = np.random.default_rng(35)
    eps = 1e-5
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        num, ana = [], []
        base = {"q": q, "k": k, "v": v}
        for _ in range(24):
            idx = tuple(int(rng.integers(0, n)) for n in base[name].shape)
            plus = {kk: a.copy() for kk, a in base.items()}
            minus = {kk: a.copy() for kk, a in base.items()}
            plus[name][idx] += eps
            minus[name][idx] -= eps
            num.append((loss(plus["q"], plus["k"], plus["v"]) -
                        loss(minus["q"], minus["k"], minus["v"])) / (2 * eps))
            ana.append(grad[idx])
        num, ana = np.array(num), np.array(ana)
        rel = np.max(np.abs(num - ana)) / max(np.max(np.abs(ana)), 1e-30)
        assert rel <= 1e-6, f"d{name}: finite-difference rel err {rel:.2e}"


# ---------------------------------------------------------------- closed forms

def pin_zero_q_uniform(orc):
    """q = 0: every visible key gets the same weight; out = mean of visible v, lse = ln |J|."""
    B, H, sq, sk, d = 2, 2, 24, 40, 8
    q_offset, key_len = 10, [40, 21]
    q = np.zeros((B, sq, H, d))
    k, v = _rand((B, sk, H, d), 41), _rand((B, sk, H, d), 42)
    out, lse = orc.attn_fwd(q, k, v, True, q_offset, key_len)
    for b in range(B):
        for i in range(sq):
            n = min(q_offset + i + 1, key_len[b])
            for h in range(H):
                assert abs(lse[b, h, i] - math.log(n)) <= 1e-13, (b, h, i)
                _close(out[b, i, h], v[b, :n, h].mean(axis=0), 1e-13, f"mean row {i}")


def pin_causal_row0(orc):
    """Causal row 0 sees only key 0: out[0] = v[0] exactly, lse[0] = scale * q0.k0."""
    B, H, S, d = 1, 3, 10, 16
    q, k, v = (_rand((B, S, H, d), 50 + t) for t in range(3))
    out, lse = orc.attn_fwd(q, k, v, True)
    for h in range(H):
        assert np.array_equal(out[0, 0, h], v[0, 0, h]), "row 0 must return v[0] exactly"
        s00 = float(np.dot(q[0, 0, h], k[0, 0, h])) / math.sqrt(d)
        assert abs(lse[0, h, 0] - s00) <= 1e-13


def pin_constant_v(orc):
    """v_j = c for all j: out_i = c (the weights sum to one)."""
    B, H, sq, sk, d = 2, 2, 17, 29, 8
    q, k = _rand((B, sq, H, d), 60, 3.0), _rand((B, sk, H, d), 61, 3.0)
    c = _rand((d,), 62)
    v = np.broadcast_to(c, (B, sk, H, d)).copy()
    for causal, off, kl in ((True, 12, None), (False, 0, [29, 5])):
        out, _ = orc.attn_fwd(q, k, v, causal, off, kl)
        _close(out, np.broadcast_to(c, out.shape), 1e-13, "constant v")


def pin_one_and_two_keys(orc):
    """One key: out = v0, lse = s0.  Two keys: weight of key 0 is logistic(s0 - s1)."""
    B, H, sq, d = 1, 2, 5, 8
    q = _rand((B, sq, H, d), 70)
    k1, v1 = _rand((B, 1, H, d), 71), _rand((B, 1, H, d), 72)
    out, lse = orc.attn_fwd(q, k1, v1, False, scale=0.7)
    for i in range(sq):
        for h in range(H):
            assert np.array_equal(out[0, i, h], v1[0, 0, h])
            assert abs(lse[0, h, i] - 0.7 * float(np.dot(q[0, i, h], k1[0, 0, h]))) <= 1e-13
    k2, v2 = _rand((B, 2, H, d), 73), _rand((B, 2, H, d), 74)
    out, lse = orc.attn_fwd(q, k2, v2, False, scale=0.7)
    for i in range(sq):
        for h in range(H):
            s0 = 0.7 * float(np.dot(q[0, i, h], k2[0, 0, h]))
            s1 = 0.7 * float(np.dot(q[0, i, h], k2[0, 1, h]))
            w0 = 1.0 / (1.0 + math.exp(s1 - s0))
            _close(out[0, i, h], w0 * v2[0, 0, h] + (1 - w0) * v2[0, 1, h], 1e-13, "two keys")
            ref_lse = max(s0, s1) + math.log1p(math.exp(-abs(s0 - s1)))
            assert abs(lse[0, h, i] - ref_lse) <= 1e-13


# ---------------------------------------------------------------- invariants

def pin_softmax_rows(orc):
    """With v_j = e_j the output row is the softmax row: non-negative, sums to 1, masked = 0."""
    B, H, sq, d = 2, 1, 12, 16
    sk = d
    q, k = _rand((B, sq, H, d), 80, 2.0), _rand((B, sk, H, d), 81, 2.0)
    v = np.zeros((B, sk, H, d))
    for j in range(sk):
        v[:, j, :, j] = 1.0
    q_offset, key_len = 2, [16, 9]
    out, _ = orc.attn_fwd(q, k, v, True, q_offset, key_len)
    for b in range(B):
        for i in range(sq):
            row = out[b, i, 0]
            n = min(q_offset + i + 1, key_len[b])
            assert abs(row.sum() - 1.0) <= 1e-13
            assert (row[:n] > 0).all() and (row[n:] == 0).all()


def pin_key_padding_is_truncation(orc):
    """Padding keys j >= L is the same problem as dropping them."""
    B, H, sq, sk, d = 1, 2, 11, 30, 8
    q, do = _rand((B, sq, H, d), 90), _rand((B, sq, H, d), 91)
    k, v = _rand((B, sk, H, d), 92), _rand((B, sk, H, d), 93)
    L = 19
    out, lse = orc.attn_fwd(q, k, v, False, key_len=[L])
    out_t, lse_t = orc.attn_fwd(q, k[:, :L], v[:, :L], False)
    _close(out, out_t, 1e-14, "out")
    _close(lse, lse_t, 1e-14, "lse")
    dq, dk, dv = orc.attn_bwd(q, k, v, do, False, key_len=[L])
    dq_t, dk_t, dv_t = orc.attn_bwd(q, k[:, :L], v[:, :L], do, False)
    _close(dq, dq_t, 1e-14, "dq")
    _close(dk[:, :L], dk_t, 1e-14, "dk")
    _close(dv[:, :L], dv_t, 1e-14, "dv")
    assert not dk[:, L:].any() and not dv[:, L:].any()


def pin_gradient_sums(orc):
    """sum_j dK_j = 0 (softmax is shift-invariant in k) and sum_j dV_j = sum_i dO_i."""
    B, H, sq, sk, d = 2, 2, 21, 21, 16
    q, do = _rand((B, sq, H, d), 100), _rand((B, sq, H, d), 101)
    k, v = _rand((B, sk, H, d), 102), _rand((B, sk, H, d), 103)
    for causal, kl in ((True, None), (False, [21, 13])):
        dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, key_len=kl)
        _close(dk.sum(axis=1), np.zeros((B, H, d)), 1e-12, "sum_j dK_j")
        _close(dv.sum(axis=1), do.sum(axis=1), 1e-12, "sum_j dV_j")


def pin_empty_rows(orc):
    """A row with no valid key: out = 0, lse = -inf, and it contributes no gradient."""
    B, H, sq, sk, d = 2, 1, 6, 9, 8
    q, do = _rand((B, sq, H, d), 110), _rand((B, sq, H, d), 111)
    k, v = _rand((B, sk, H, d), 112), _rand((B, sk, H, d), 113)
    out, lse = orc.attn_fwd(q, k, v, False, key_len=[0, 9])
    assert not out[0].any() and np.all(np.isneginf(lse[0]))
    dq, dk, dv = orc.attn_bwd(q, k, v, do, False, key_len=[0, 9])
    assert not dq[0].any() and not dk[0].any() and not dv[0].any()


def pin_rows_api(orc):
    """The row-range entry points agree with the full-tensor ones."""
    B, H, sq, sk, d = 2, 2, 40, 64, 8
    q, do = _rand((B, sq, H, d), 120), _rand((B, sq, H, d), 121)
    k, v = _rand((B, sk, H, d), 122), _rand((B, sk, H, d), 123)
    off, kl = 24, [64, 50]
    out, lse = orc.attn_fwd(q, k, v, True, off, kl)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, True, off, kl)
    for (b, h, i0, i1, j0, j1) in ((0, 1, 3, 17, 40, 64), (1, 0, 0, 40, 0, 5)):
        o, l = orc.attn_fwd_rows(q, k, v, b, h, i0, i1, True, off, kl)
        _close(o, out[b, i0:i1, h], 1e-14, "rows out")
        _close(l, lse[b, h, i0:i1], 1e-14, "rows lse")
        rq, rk, rv = orc.attn_bwd_rows(q, k, v, do, b, h, i0, i1, j0, j1, True, off, kl)
        _close(rq, dq[b, i0:i1, h], 1e-14, "rows dq")
        _close(rk, dk[b, j0:j1, h], 1e-14, "rows dk")
        _close(rv, dv[b, j0:j1, h], 1e-14, "rows dv")


# ---------------------------------------------------------------- the pages' worked examples

def _read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def pin_golden_causal_example(orc):
    """adv07 tutorial section 3 Q4: seq 1024 on 2 cards; row i (global) sees i+1 keys."""
    d = 4
    for seq, sp, shard, first, grow, nvis in (tuple(map(int, r)) for r in _read_rows(
            "sp_tutorial_causal_example.txt")):
        sq = seq // sp
        q = np.zeros((1, sq, 1, d))
        k = _rand((1, seq, 1, d), 130)
        v = _rand((1, seq, 1, d), 131)
        i = grow - first
        out, lse = orc.attn_fwd_rows(q, k, v, 0, 0, i, i + 1, True, q_offset=first)
        assert abs(lse[0] - math.log(nvis)) <= 1e-12, (grow, lse[0], math.log(nvis))
        _close(out[0], v[0, :nvis, 0].mean(axis=0), 1e-12, f"row {grow}")


def pin_golden_split_q(orc):
    """adv07 tutorial sections 4 and 6: Q shards against the full K/V, concatenated,
    equal unsharded attention (printed bound: max abs error < 1e-5)."""
    for seq, d, splits, bound in ((int(a), int(b), int(c), float(e)) for a, b, c, e in _read_rows(
            "sp_tutorial_split_q.txt")):
        q, k, v = (_rand((1, seq, 1, d), 140 + t) for t in range(3))
        chunk = (seq + splits - 1) // splits
        for causal in (False, True):
            full, _ = orc.attn_fwd(q, k, v, causal)
            parts = []
            for s in range(splits):
                lo, hi = s * chunk, min((s + 1) * chunk, seq)
                o, _ = orc.attn_fwd(q[:, lo:hi], k, v, causal, q_offset=lo)
                parts.append(o)
            err = float(np.max(np.abs(np.concatenate(parts, axis=1) - full)))
            assert err < bound and err <= 1e-13, (seq, splits, causal, err)


def pin_negative_control(orc):
    """adv07 tutorial section 4: shards that only see their own K/V are NOT attention."""
    seq, d = 16, 32
    q, k, v = (_rand((1, seq, 1, d), 150 + t) for t in range(3))
    full, _ = orc.attn_fwd(q, k, v, True)
    wrong = []
    for lo, hi in ((0, 8), (8, 16)):
        o, _ = orc.attn_fwd(q[:, lo:hi], k[:, lo:hi], v[:, lo:hi], True)
        wrong.append(o)
    err = float(np.max(np.abs(np.concatenate(wrong, axis=1) - full)))
    assert err > 1e-2, f"own-shard K/V should differ from full attention, got {err:.2e}"
    assert np.max(np.abs(wrong[0] - full[:, :8])) <= 1e-14   # shard 0 is unaffected


def pin_relayout_golden(orc):
    """Hand-derived regrouping cases (fixture relayout_worked_examples.txt)."""
    rows = _read_rows("relayout_worked_examples.txt")
    for n in range(0, len(rows), 3):
        assert rows[n][0] == "case" and rows[n + 1][0] == "in" and rows[n + 2][0] == "out"
        N, b, s, h, d = map(int, rows[n][1:])
        x = np.array(list(map(int, rows[n + 1][1:])), dtype=np.uint16)
        y = np.array(list(map(int, rows[n + 2][1:])), dtype=np.uint16)
        got = orc.seq2head(x, N, b, s, h, d).reshape(-1)
        assert np.array_equal(got, y), (rows[n], got, y)
        back = orc.head2seq(y, N, b, s, h, d).reshape(-1)
        assert np.array_equal(back, x), (rows[n], back, x)


def pin_relayout_torch(orc):
    """seq->head equals torch's view/permute of the concatenated sequence; round trip is exact."""
    for (N, b, s, h, d) in ((2, 1, 8, 2, 4), (4, 2, 12, 8, 3), (8, 1, 16, 16, 2), (1, 3, 5, 2, 2)):
        x = torch.randint(0, 65535, (N, b, s // N, h, d), dtype=torch.int32).to(torch.int16)
        full = x.permute(1, 0, 2, 3, 4).reshape(b, s, h, d)
        ref = full.reshape(b, s, N, h // N, d).permute(2, 0, 1, 3, 4).contiguous()
        got = orc.seq2head(x.numpy(), N, b, s, h, d)
        assert np.array_equal(got, ref.numpy().view(np.uint16)), (N, b, s, h, d)
        back = orc.head2seq(got, N, b, s, h, d)
        assert np.array_equal(back, x.numpy().view(np.uint16))


def _chunk_key_len(key_len, lo, hi):
    """Valid keys of chunk [lo, hi) given the full key_len per batch entry."""
    if key_len is None:
        return None
    return [min(max(n - lo, 0), hi - lo) for n in key_len]


def pin_merge_split_kv(orc):
    """adv07 tutorial sections 5 and 7 (ring / blockwise attention): attention against
    each key chunk, the query position taken relative to the chunk's first key, merged by
    the log-sum-exp rule equals attention against all keys.  Chunks are ragged; some
    rows see no key of a chunk, and one batch entry has no visible key at all."""
    B, H, sq, sk, d = 2, 2, 23, 41, 8
    q, k, v = _rand((B, sq, H, d), 170), _rand((B, sk, H, d), 171), _rand((B, sk, H, d), 172)
    bounds = [(0, 7), (7, 20), (20, 33), (33, 41)]
    for causal, q_offset, key_len in ((True, 18, None), (True, 0, [41, 0]),
                                      (False, 0, [41, 12]), (False, 0, None)):
        full, full_lse = orc.attn_fwd(q, k, v, causal, q_offset, key_len)
        outs, lses = [], []
        for lo, hi in bounds:
            o, l = orc.attn_fwd(q, k[:, lo:hi], v[:, lo:hi], causal, q_offset - lo,
                                _chunk_key_len(key_len, lo, hi))
            outs.append(o)
            lses.append(l)
        out, lse = orc.attn_merge(outs, lses)
        _close(out, full, 1e-12, f"merged out causal={causal}")
        fin = np.isfinite(full_lse)
        assert np.array_equal(np.isfinite(lse), fin)
        _close(lse[fin], full_lse[fin], 1e-12, f"merged lse causal={causal}")
        # merging is order-free
        rev, rev_lse = orc.attn_merge(outs[::-1], lses[::-1])
        _close(rev, out, 1e-13, "merge order")


def pin_merge_closed_forms(orc):
    """Two copies of one result: same out, lse + ln 2.  An empty partial (lse = -inf)
    changes nothing.  All partials empty: out 0, lse -inf."""
    B, H, sq, d = 1, 2, 5, 4
    o = _rand((B, sq, H, d), 180)
    lse = _rand((B, H, sq), 181)
    out, l2 = orc.attn_merge([o, o], [lse, lse])
    _close(out, o, 1e-14, "duplicate out")
    _close(l2, lse + math.log(2.0), 1e-14, "duplicate lse")
    empty_lse = np.full_like(lse, -np.inf)
    out, l1 = orc.attn_merge([o, np.zeros_like(o)], [lse, empty_lse])
    assert np.array_equal(out, o) and np.array_equal(l1, lse)
    out, l0 = orc.attn_merge([np.zeros_like(o)] * 2, [empty_lse, empty_lse])
    assert not out.any() and np.all(l0 == -np.inf)


def pin_linear_loops(orc):
    """nn.Linear y = x W^T, dx = dy W, dW = dy^T x against explicit loops on tiny shapes
    ("Parallel multi-head attention", sections 2.1 and 2.3: Column/RowParallelLinear)."""
    import oracle as om
    M, n_in, n_out = 5, 4, 3
    x, w, dy = _rand((M, n_in), 210), _rand((n_out, n_in), 211), _rand((M, n_out), 212)
    y = om.linear_fwd(x, w)
    dx, dw = om.linear_bwd(dy, x, w)
    for i in range(M):
        for o in range(n_out):
            assert abs(y[i, o] - sum(x[i, c] * w[o, c] for c in range(n_in))) <= 1e-13
        for c in range(n_in):
            assert abs(dx[i, c] - sum(dy[i, o] * w[o, c] for o in range(n_out))) <= 1e-13
    for o in range(n_out):
        for c in range(n_in):
            assert abs(dw[o, c] - sum(dy[i, o] * x[i, c] for i in range(M))) <= 1e-13


def pin_layer_identity_weights(orc):
    """Identity projections (wq = wk = wv = wo = I): the layer is attention of the shards
    with themselves as q, k and v, regrouped by the oracle's own seq->head formula."""
    import oracle as om
    N, b, s, h, d = 2, 1, 12, 4, 4
    dim = h * d
    x = _rand((N, b, s // N, dim), 220)
    eye = np.eye(dim)
    L = om.Layer(orc, N, h, d)
    out = L.forward(x, np.concatenate([eye, eye, eye]), eye)
    shards = x.reshape(N, b, s // N, h, d)
    groups = om._groups_of(shards, N)
    ref = np.empty_like(groups)
    for g in range(N):
        ref[g], _ = orc.attn_fwd(groups[g], groups[g], groups[g], True)
    _close(out, om._shards_of(ref, N).reshape(x.shape), 1e-13, "identity-weight layer")
    # the float regrouping agrees with the pinned 16-bit one
    bits = np.arange(shards.size, dtype=np.uint16).reshape(shards.shape)
    assert np.array_equal(om._groups_of(bits.astype(np.float64), N).astype(np.uint16),
                          orc.seq2head(bits, N, b, s, h, d))


def pin_layer_finite_differences(orc):
    """Central differences of sum(dout * layer(x)) for dx, dWqkv and dWo."""
    import oracle as om
    N, b, s, h, d = 2, 1, 8, 2, 4
    dim = 8
    x = _rand((N, b, s // N, dim), 230)
    wqkv, wo = _rand((3 * h * d, dim), 231, 0.5), _rand((dim, h * d), 232, 0.5)
    dout = _rand((N, b, s // N, dim), 233)
    L = om.Layer(orc, N, h, d)
    L.forward(x, wqkv, wo)
    dx, dwqkv, dwo = L.backward(dout)
    eps = 1e-6
    rng = np.random.default_rng(234)
    for arr, grad, name in ((x, dx, "dx"), (wqkv, dwqkv, "dwqkv"), (wo, dwo, "dwo")):
        for _ in range(6):
            idx = tuple(rng.integers(0, n) for n in arr.shape)
            old = arr[idx]
            arr[idx] = old + eps
            f1 = float(np.sum(dout * om.Layer(orc, N, h, d).forward(x, wqkv, wo)))
            arr[idx] = old - eps
            f0 = float(np.sum(dout * om.Layer(orc, N, h, d).forward(x, wqkv, wo)))
            arr[idx] = old
            num = (f1 - f0) / (2 * eps)
            assert abs(num - grad[idx]) <= 1e-6 * max(1.0, abs(num)), (name, idx, num, grad[idx])


ALL_PINS = [
    pin_sdpa_causal_square, pin_sdpa_masks, pin_finite_differences, pin_zero_q_uniform,
    pin_causal_row0, pin_constant_v, pin_one_and_two_keys, pin_softmax_rows,
    pin_key_padding_is_truncation, pin_gradient_sums, pin_empty_rows, pin_rows_api,
    pin_golden_causal_example, pin_golden_split_q, pin_negative_control,
    pin_relayout_golden, pin_relayout_torch, pin_merge_split_kv, pin_merge_closed_forms,
    pin_sdpa_key_mask, pin_key_mask_special_cases, pin_linear_loops,
    pin_layer_identity_weights, pin_layer_finite_differences,
]
