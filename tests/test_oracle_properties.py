"""Property tests of the fp64 oracle on generated small problems (hypothesis, derandomised
so that every run draws the same cases).

Each property ties the oracle to something outside itself over many shapes at once,
beside the fixed cases of oracle_pins.py:
  * attention forward and backward equal torch's fp64 scaled_dot_product_attention with
    an explicit boolean mask and its autograd derivative, for any mix of causal masking,
    query offset (a query shard's global position, "adv07: Sequence Parallel" section 3
    Q4), right-padded key lengths, a general key mask (PR 31525's attention_mask =
    input_ids != pad) and softmax scale, empty rows included;
  * attention against key chunks merged by the log-sum-exp rule equals attention against
    all keys (ring / blockwise attention, adv07 sections 5 and 7), for any chunking;
  * the regrouping equals torch's reshape/permute of the concatenated sequence and its
    inverse restores the shards bit for bit.
"""
import math

import numpy as np
import torch
from hypothesis import HealthCheck, given, settings
from hypothesis import strategies as st

import oracle
from oracle_pins import _chunk_key_len, _torch_reference

SETTINGS = settings(max_examples=60, deadline=None, derandomize=True,
                    suppress_health_check=[HealthCheck.too_slow])


@st.composite
def problems(draw):
    B = draw(st.integers(1, 3))
    H = draw(st.integers(1, 3))
    sq = draw(st.integers(1, 20))
    sk = draw(st.integers(1, 24))
    d = draw(st.integers(1, 12))
    causal = draw(st.booleans())
    q_offset = draw(st.integers(0, 24)) if causal else 0
    key_len = draw(st.one_of(st.none(), st.lists(st.integers(0, sk), min_size=B, max_size=B)))
    key_mask = draw(st.one_of(st.none(), st.lists(
        st.lists(st.booleans(), min_size=sk, max_size=sk), min_size=B, max_size=B)))
    scale = draw(st.one_of(st.none(), st.floats(0.05, 2.0)))
    seed = draw(st.integers(0, 2 ** 31 - 1))
    return B, H, sq, sk, d, causal, q_offset, key_len, key_mask, scale, seed


def check_attention(orc, case):
    """Forward and backward of one generated problem against torch fp64 sdpa + autograd."""
    B, H, sq, sk, d, causal, q_offset, key_len, key_mask, scale, seed = case
    rng = np.random.default_rng(seed)
    q, do = (rng.standard_normal((B, sq, H, d)) for _ in range(2))
    k, v = (rng.standard_normal((B, sk, H, d)) for _ in range(2))
    mask = None if key_mask is None else np.asarray(key_mask, dtype=np.uint8)
    out, lse = orc.attn_fwd(q, k, v, causal, q_offset, key_len, scale, key_mask=mask)
    dq, dk, dv = orc.attn_bwd(q, k, v, do, causal, q_offset, key_len, scale, key_mask=mask)
    s = 1.0 / math.sqrt(d) if scale is None else scale
    r_out, r_lse, r_dq, r_dk, r_dv, rows_ok = _torch_reference(q, k, v, do, causal, q_offset,
                                                               key_len, s, mask)
    np.testing.assert_allclose(out, r_out, rtol=0, atol=1e-11)
    np.testing.assert_allclose(dq, r_dq, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dk, r_dk, rtol=0, atol=1e-10)
    np.testing.assert_allclose(dv, r_dv, rtol=0, atol=1e-10)
    fin = np.isfinite(r_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], r_lse[fin], rtol=0, atol=1e-11)
    assert np.all(lse[~fin] == -np.inf)
    # rows with no visible key ([B][sq], the mask is per batch entry): out 0, no dq
    empty = ~rows_ok
    assert not out[empty].any() and not dq[empty].any()


@SETTINGS
@given(problems())
def test_attention_equals_torch_sdpa_and_autograd(case):
    check_attention(oracle.default(), case)


@st.composite
def chunkings(draw):
    B, H, sq, sk, d, causal, q_offset, key_len, _, scale, seed = draw(problems())
    cuts = sorted(set(draw(st.lists(st.integers(1, max(sk - 1, 1)), max_size=4))) - {sk})
    bounds = list(zip([0] + cuts, cuts + [sk]))
    return B, H, sq, sk, d, causal, q_offset, key_len, scale, seed, bounds


def check_merge(orc, case):
    """Per-chunk attention merged by the log-sum-exp rule against attention over all keys."""
    B, H, sq, sk, d, causal, q_offset, key_len, scale, seed, bounds = case
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, sq, H, d))
    k, v = (rng.standard_normal((B, sk, H, d)) for _ in range(2))
    full, full_lse = orc.attn_fwd(q, k, v, causal, q_offset, key_len, scale)
    outs, lses = [], []
    for lo, hi in bounds:
        # the chunk's keys, the query position taken relative to its first key (negative
        # when the chunk starts after a row's position: that row sees none of it)
        o, l = orc.attn_fwd(q, k[:, lo:hi], v[:, lo:hi], causal, q_offset - lo,
                            _chunk_key_len(key_len, lo, hi), scale)
        outs.append(o)
        lses.append(l)
    out, lse = orc.attn_merge(outs, lses)
    np.testing.assert_allclose(out, full, rtol=0, atol=1e-11)
    fin = np.isfinite(full_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], full_lse[fin], rtol=0, atol=1e-11)


@SETTINGS
@given(chunkings())
def test_split_kv_merge_equals_full_attention(case):
    check_merge(oracle.default(), case)


regroupings = st.tuples(st.integers(1, 6), st.integers(1, 3), st.integers(1, 5),
                        st.integers(1, 4), st.integers(1, 6), st.integers(0, 2 ** 31 - 1))


def check_regrouping(orc, case):
    """seq->head against torch's reshape/permute; head->seq restores the shards."""
    N, b, sl, hl, d, seed = case
    s, h = N * sl, N * hl
    g = torch.Generator().manual_seed(seed)
    x = torch.randint(-32768, 32767, (N, b, sl, h, d), generator=g, dtype=torch.int32)
    x = x.to(torch.int16)
    got = orc.seq2head(x.numpy(), N, b, s, h, d)
    full = x.permute(1, 0, 2, 3, 4).reshape(b, s, h, d)          # shards in sequence order
    ref = full.reshape(b, s, N, hl, d).permute(2, 0, 1, 3, 4)     # head group g first
    assert np.array_equal(got, ref.contiguous().numpy().view(np.uint16))
    assert np.array_equal(orc.head2seq(got, N, b, s, h, d), x.numpy().view(np.uint16))


@SETTINGS
@given(regroupings)
def test_regrouping_equals_torch_permute(case):
    check_regrouping(oracle.default(), case)


# (strategy, check) pairs, for the mutant test: a broken oracle must fail one of them
PROPERTIES = [(problems(), check_attention), (chunkings(), check_merge),
              (regroupings, check_regrouping)]
