"""GPU relayout against the oracle's index loop: bit-exact, every workload shape
plus odd shapes (narrow runs, one shard, many tensors per launch)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_status, need_gpu, u16
from sequence_head_attention_seq_b300 import (sp_relayout_head2seq, sp_relayout_seq2head,
                                              workloads)

pytestmark = pytest.mark.gpu


def _rand_bits(shape, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return torch.randint(-32768, 32767, shape, generator=g, device="cuda",
                         dtype=torch.int32).to(torch.int16).view(torch.bfloat16)


@pytest.mark.parametrize("N,b,s,h,d", [
    (2, 1, 128, 2, 64),       # two shards, one head per group
    (4, 2, 64, 8, 128),
    (8, 1, 256, 64, 128),
    (3, 2, 12, 6, 8),         # run = 2*8 elements (16-byte vectors)
    (2, 3, 10, 2, 2),         # run = 2 elements (4-byte path)
    (2, 1, 6, 2, 1),          # run = 1 element (2-byte path)
    (1, 2, 16, 4, 64),        # one shard: a plain copy
])
def test_relayout_matches_oracle(N, b, s, h, d):
    need_gpu()
    orc = oracle.default()
    xs = [_rand_bits((N, b, s // N, h, d), 100 + t) for t in range(3)]
    groups = sp_relayout_seq2head(xs, N)
    back = sp_relayout_head2seq(groups, N)
    torch.cuda.synchronize()
    check_status()
    for x, g, y in zip(xs, groups, back):
        ref = orc.seq2head(u16(x), N, b, s, h, d)
        assert np.array_equal(u16(g), ref)
        assert np.array_equal(u16(y), u16(x))
        assert np.array_equal(orc.head2seq(u16(g), N, b, s, h, d), u16(x))


def test_eight_tensors_in_one_launch():
    need_gpu()
    N, b, s, h, d = 4, 1, 32, 8, 64
    xs = [_rand_bits((N, b, s // N, h, d), 200 + t) for t in range(8)]
    outs = sp_relayout_seq2head(xs, N)
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()
    for x, o in zip(xs, outs):
        assert np.array_equal(u16(o), orc.seq2head(u16(x), N, b, s, h, d))


@pytest.mark.parametrize("name", [w for w in workloads.ORDER if workloads.WORKLOADS[w].N > 1])
def test_relayout_workloads(name):
    """Every workload's Q/K/V shards through seq->head and back, against the oracle."""
    need_gpu()
    w = workloads.WORKLOADS[name]
    ins = workloads.make_inputs(w, device="cuda", with_dout=False)
    xs = [ins["q"], ins["k"], ins["v"]]
    groups = sp_relayout_seq2head(xs, w.N)
    back = sp_relayout_head2seq(groups, w.N)
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()
    # the oracle's scalar loop on the first tensor; all three must round-trip exactly
    ref = orc.seq2head(u16(xs[0]), w.N, w.b, w.s, w.h, w.d)
    assert np.array_equal(u16(groups[0]), ref)
    del ref
    for x, y in zip(xs, back):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))
    for x, g in zip(xs[1:], groups[1:]):
        # K/V: spot rows of every group against the oracle's definition
        for gi in (0, w.N - 1):
            for t in (0, w.s_local - 1, w.s_local, w.s - 1):
                r, u = divmod(t, w.s_local)
                got = g[gi, 0, t].view(torch.int16)
                want = x[r, 0, u, gi * w.h_local:(gi + 1) * w.h_local].view(torch.int16)
                assert torch.equal(got, want)


@pytest.mark.parametrize("N,b,s,h,d", [
    (2, 1, 128, 2, 64),
    (4, 2, 64, 8, 128),
    (3, 2, 12, 6, 8),
    (2, 3, 10, 4, 2),         # 4-byte runs; each part starts 16 bytes into the row
])
def test_packed_relayout_matches_oracle(N, b, s, h, d):
    """Packed [N][b][s/N][3][h][d] shards: each of the three parts regrouped exactly as the
    oracle regroups it alone, and the packed inverse restores the buffer bit for bit."""
    need_gpu()
    orc = oracle.default()
    qkv = _rand_bits((N, b, s // N, 3, h, d), 300 + s)
    from sequence_head_attention_seq_b300 import (sp_relayout_head2seq_packed,
                                                  sp_relayout_seq2head_packed)
    groups = sp_relayout_seq2head_packed(qkv, N)
    back = sp_relayout_head2seq_packed(groups, N)
    torch.cuda.synchronize()
    check_status()
    for t in range(3):
        part = qkv[:, :, :, t].contiguous()
        assert np.array_equal(u16(groups[t]), orc.seq2head(u16(part), N, b, s, h, d)), t
    assert np.array_equal(u16(back), u16(qkv))


@pytest.mark.parametrize("N,b,s,h,d", [(2, 1, 128, 2, 64), (4, 2, 64, 8, 128), (3, 2, 12, 6, 8)])
def test_all_to_all_form_matches_oracle(N, b, s, h, d):
    """sp_relayout with (scatter 2, gather 1) and (scatter 1, gather 2): the oracle's
    index loop, bit for bit, and the inverse of each other."""
    need_gpu()
    from sequence_head_attention_seq_b300 import sp_relayout
    orc = oracle.default()
    x = _rand_bits((N, b, s // N, h, d), 300 + N)
    g = sp_relayout(x, N, 2, 1)
    y = sp_relayout(g, N, 1, 2)
    torch.cuda.synchronize()
    check_status()
    assert tuple(g.shape) == (N, b, s, h // N, d)
    assert np.array_equal(u16(g), orc.seq2head(u16(x), N, b, s, h, d))
    assert np.array_equal(u16(y), u16(x))
