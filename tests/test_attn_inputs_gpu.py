"""GPU attention against the fp64 oracle on inputs the workload-shaped tests do not
reach: scores that grow along the key sequence (so that the forward's running maximum
moves by more than its lazy-rescale threshold and O is rescaled in TMEM), an explicit
softmax scale, and tensors that are strided views rather than contiguous buffers.

What is computed is the same as in the other parity tests ("adv07: Sequence Parallel",
section 3 Q4; "Parallel multi-head attention", section 3.2: softmax(q k^T * scale) v
over the visible keys, scale = 1/sqrt(head_dim) unless given); the bars are the same
(out max-abs 1e-2 / mean-abs 1e-3, lse 1e-2, gradients relative Frobenius 2e-2), except
that the explicit-scale cases add each output's own bf16 rounding (2^-8 of its
magnitude) to the max-abs bar, because a peaked softmax gives outputs of magnitude 2 to 4
(see `_check_out_rounded`)."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_lse, check_out, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import sp_attn_bwd, sp_attn_fwd, workloads

pytestmark = pytest.mark.gpu

# the forward rescales O only when a row's maximum grows by more than this many
# log2 units; the inputs below are checked to cross it with a margin
RESCALE_LOG2 = 8.0


def _randn(shape, seed, scale=1.0):
    return workloads.randn_bf16(shape, seed, scale, device="cuda")


def _check_out_rounded(gpu: np.ndarray, ref: np.ndarray, what: str):
    """The output bar with the bf16 output's own rounding added: |gpu - oracle| <= 1e-2 +
    2^-8 |oracle| element by element (half a bf16 unit in the last place is at most
    2^-8 of the value), and the mean-abs bar unchanged.  A peaked softmax (a large
    scale) gives outputs close to single v rows, of magnitude 2 to 4, where rounding to
    bf16 alone moves a value by up to 2^-7 and the absolute bar would measure the
    output format rather than the kernel."""
    err = np.abs(gpu - ref)
    bound = 1e-2 + 2.0 ** -8 * np.abs(ref)
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (f"{what}: {int((err > bound).sum())} elements off, worst "
                                  f"{err[worst]:.3e} at |oracle| {abs(ref[worst]):.3f}")
    assert err.mean() <= 1e-3, f"{what}: mean abs {err.mean():.3e}"


def _compare(q, k, v, do, causal, q_offset=0, key_len=None, scale=None, o=None, lse=None,
             out_check=check_out):
    """Run forward and backward through the library and compare every output with the
    oracle on the same bf16 inputs."""
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device="cuda")
    o, lse = sp_attn_fwd(q, k, v, causal, q_offset, kl, softmax_scale=scale, out=o, lse=lse)
    dq, dk, dv = sp_attn_bwd(q, k, v, o, lse, do, causal, q_offset, kl, softmax_scale=scale)
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()
    ro, rl = orc.attn_fwd(f64(q), f64(k), f64(v), causal, q_offset, key_len, scale)
    rdq, rdk, rdv = orc.attn_bwd(f64(q), f64(k), f64(v), f64(do), causal, q_offset, key_len,
                                 scale)
    out_check(f64(o), ro, "out")
    check_lse(f64(lse), rl, "lse")
    check_grad(f64(dq), rdq, "dq")
    check_grad(f64(dk), rdk, "dk")
    check_grad(f64(dv), rdv, "dv")
    return o, lse, dq, dk, dv


def _trend_inputs(B, H, s, d, seed):
    """q, k, v, dout ~ N(0, 1) with one coordinate replaced by a trend: k[j, 0] grows by
    `step` per 128-key block and q[i, 0] is 0, 4 or 8 by row (i % 3), so the scores of a
    row with q[i, 0] = 8 rise by about 8 natural units (11.5 log2 units) per key block,
    those of q[i, 0] = 4 by half that and those of q[i, 0] = 0 not at all.  Every value
    written is exact in bf16."""
    q = _randn((B, s, H, d), seed)
    k = _randn((B, s, H, d), seed + 1)
    v = _randn((B, s, H, d), seed + 2)
    do = _randn((B, s, H, d), seed + 3)
    step = 8.0 if d == 64 else 12.0          # 8 * step / sqrt(d) = 8 or 8.49 per block
    blk = torch.arange(s, device="cuda") // 128
    k[:, :, :, 0] = (step * blk).to(torch.bfloat16).view(1, s, 1)
    c = torch.tensor([0.0, 4.0, 8.0], device="cuda")[torch.arange(s, device="cuda") % 3]
    q[:, :, :, 0] = c.to(torch.bfloat16).view(1, s, 1)
    return q, k, v, do


def _rescaling_rows(q, k, causal, key_len, scale):
    """Fraction of rows whose running maximum of scaled scores (log2 units, over key
    blocks of 128 in order) ever grows by more than the threshold plus a margin, and the
    fraction whose maximum never grows by more than the threshold minus a margin."""
    qf, kf = f64(q), f64(k)
    B, s, H, d = qf.shape
    sk = kf.shape[1]
    up = never = total = 0
    for b in range(B):
        n = sk if key_len is None else key_len[b]
        for h in range(H):
            sc = (qf[b, :, h] @ kf[b, :n, h].T) * scale * math.log2(math.e)
            if causal:
                sc = np.where(np.arange(n)[None, :] <= np.arange(s)[:, None], sc, -np.inf)
            nb = (n + 127) // 128
            blk = np.stack([sc[:, 128 * j:128 * (j + 1)].max(axis=1) for j in range(nb)], 1)
            run = np.maximum.accumulate(blk, axis=1)
            with np.errstate(invalid="ignore"):
                jump = np.where(np.isfinite(run[:, :-1]), blk[:, 1:] - run[:, :-1], 0.0)
            jump = np.nan_to_num(jump, nan=0.0, neginf=0.0)
            mx = jump.max(axis=1) if nb > 1 else np.zeros(s)
            up += int((mx > RESCALE_LOG2 + 1.0).sum())
            never += int((mx < RESCALE_LOG2 - 1.0).sum())
            total += s
    return up / total, never / total


RESCALE = [
    # B, H, s, d, causal, key_len
    (1, 2, 640, 64, True, None),
    (1, 2, 640, 128, True, None),
    (2, 1, 640, 128, False, [640, 300]),
    (1, 3, 520, 64, False, None),
]


@pytest.mark.parametrize("case", RESCALE, ids=[str(c) for c in RESCALE])
def test_growing_scores_rescale_the_running_maximum(case):
    """Online softmax with O rescaled in TMEM: within one warp some rows rescale at
    every key block and others never do; the result must still equal the oracle's
    plain softmax over all visible keys."""
    need_gpu()
    B, H, s, d, causal, key_len = case
    q, k, v, do = _trend_inputs(B, H, s, d, 500 + s + d)
    up, never = _rescaling_rows(q, k, causal, key_len, 1.0 / math.sqrt(d))
    assert up >= 0.15 and never >= 0.25, (up, never)
    _compare(q, k, v, do, causal, 0, key_len)


SCALES = [
    # B, H, sq, sk, d, causal, q_offset, key_len, softmax_scale
    (2, 2, 300, 300, 128, True, 0, None, 0.02),
    (1, 3, 200, 456, 64, False, 0, [400], 0.4),
    (1, 2, 260, 516, 128, True, 256, None, 0.25),
]


@pytest.mark.parametrize("case", SCALES, ids=[str(c) for c in SCALES])
def test_explicit_softmax_scale(case):
    """softmax_scale given by the caller instead of 1/sqrt(head_dim).  With scale 0.4 at
    d = 64 the scores have a standard deviation of about 3.2, so some outputs reach
    magnitude 2 to 4 and the output bar includes their bf16 rounding."""
    need_gpu()
    B, H, sq, sk, d, causal, q_offset, key_len, scale = case
    seed = 31 * sq + sk
    q = _randn((B, sq, H, d), seed)
    k = _randn((B, sk, H, d), seed + 1)
    v = _randn((B, sk, H, d), seed + 2)
    do = _randn((B, sq, H, d), seed + 3)
    _compare(q, k, v, do, causal, q_offset, key_len, scale, out_check=_check_out_rounded)


def test_views_of_a_packed_qkv_buffer():
    """q, k, v as views of one [B][s][3][H][d] buffer (sequence stride 3*H*d); dq, dk, dv
    come back with the same strides."""
    need_gpu()
    B, s, H, d = 2, 384, 3, 64
    qkv = _randn((B, s, 3, H, d), 71)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    assert not q.is_contiguous()
    do = _randn((B, s, H, d), 72)
    _, _, dq, dk, dv = _compare(q, k, v, do, True)
    assert dq.stride() == q.stride() and dk.stride() == k.stride() and dv.stride() == v.stride()


def test_head_major_views():
    """Tensors stored head-major ([B][H][s][d], the layout of a transposed projection
    output) and passed as [B][s][H][d] views (sequence stride d, head stride s*d); out
    and dout in the same layout."""
    need_gpu()
    B, H, sq, sk, d = 2, 2, 333, 333, 128
    q = _randn((B, H, sq, d), 81).transpose(1, 2)
    k = _randn((B, H, sk, d), 82).transpose(1, 2)
    v = _randn((B, H, sk, d), 83).transpose(1, 2)
    do = _randn((B, H, sq, d), 84).transpose(1, 2)
    o = torch.empty((B, H, sq, d), dtype=torch.bfloat16, device="cuda").transpose(1, 2)
    _compare(q, k, v, do, True, o=o)
    _compare(q, k, v, do, False, key_len=[333, 129], o=o)


def test_mixed_layouts():
    """Each tensor with its own strides: q a view of a packed buffer, k contiguous, v
    head-major."""
    need_gpu()
    B, sq, sk, H, d = 1, 300, 420, 4, 128
    q = _randn((B, sq, 3, H, d), 91)[:, :, 1]
    k = _randn((B, sk, H, d), 92)
    v = _randn((B, H, sk, d), 93).transpose(1, 2)
    do = _randn((B, sq, H, d), 94)
    _compare(q, k, v, do, True, q_offset=120)
