"""The Ulysses regrouping fused into the attention kernels' addressing (q, k, v, o and
their gradients read and written in the sequence-shard layout [N][b][s/N][h][d], no
relayout launches) against the step with the two explicit relayouts: the same kernels,
the same arithmetic in the same order, so the forward and dK/dV are identical bit for
bit and dQ (whose fp32 additions happen in any order) agrees within the gradient bar."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_lse, check_out, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import SpError, UlyssesAttention, sp_attn_fwd, workloads

pytestmark = pytest.mark.gpu


def _both(w):
    ins = workloads.make_inputs(w, device="cuda")
    kl = ins["key_len"]
    res = []
    for fused in (False, True):
        step = UlyssesAttention(w.N, w.b, w.s, w.h, w.d, w.causal, key_len=kl, fused=fused)
        o = step.forward(ins["q"], ins["k"], ins["v"]).clone()
        lse = step.lse.clone()
        grads = [t.clone() for t in step.backward(ins["dout"])]
        torch.cuda.synchronize()
        check_status()
        res.append((o, lse, grads))
        del step
    return ins, res


SHAPES = [
    workloads.Workload("shards2", 90, b=2, h=4, d=64, s=512, N=2, causal=True, scale=1.0),
    workloads.Workload("shards4_pad", 91, b=2, h=8, d=128, s=2048, N=4, causal=False, scale=1.0,
                       key_len_range=(700, 2048)),
    workloads.WORKLOADS["llama7b"],
    workloads.WORKLOADS["llama70b"],
]


@pytest.mark.parametrize("w", SHAPES, ids=[w.name for w in SHAPES])
def test_fused_layout_equals_relayout_path(w):
    need_gpu()
    _, ((o0, l0, g0), (o1, l1, g1)) = _both(w)
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)), "out"
    assert torch.equal(l0, l1), "lse"
    for name, a, b in zip(("dk", "dv"), g0[1:], g1[1:]):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
    check_grad(f64(g1[0]), f64(g0[0]), "dq")


def test_fused_layout_against_oracle():
    """One head group of a fused step, regrouped by the oracle, against the oracle."""
    need_gpu()
    w = SHAPES[0]
    ins = workloads.make_inputs(w, device="cuda")
    step = UlyssesAttention(w.N, w.b, w.s, w.h, w.d, w.causal, fused=True)
    o = step.forward(ins["q"], ins["k"], ins["v"])
    dq, dk, dv = step.backward(ins["dout"])
    torch.cuda.synchronize()
    check_status()
    orc = oracle.default()

    def groups(t):
        bits = t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        g = orc.seq2head(bits, w.N, w.b, w.s, w.h, w.d)
        return torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16).double().numpy()

    q, k, v, do = (groups(ins[n]) for n in ("q", "k", "v", "dout"))
    og, dqg, dkg, dvg = (groups(t) for t in (o, dq, dk, dv))
    for g in range(w.N):
        ro, rl = orc.attn_fwd(q[g], k[g], v[g], w.causal)
        rdq, rdk, rdv = orc.attn_bwd(q[g], k[g], v[g], do[g], w.causal)
        check_out(og[g], ro, f"group {g} out")
        check_lse(step.lse[g * w.b:(g + 1) * w.b].double().cpu().numpy(), rl, f"group {g} lse")
        check_grad(dqg[g], rdq, f"group {g} dq")
        check_grad(dkg[g], rdk, f"group {g} dk")
        check_grad(dvg[g], rdv, f"group {g} dv")


MASKED = [
    # N, b, s, h, d, causal
    (2, 2, 512, 4, 64, True),
    (4, 1, 1024, 8, 128, False),
]


@pytest.mark.parametrize("case", MASKED, ids=[str(c) for c in MASKED])
def test_fused_layout_with_key_mask(case):
    """A general key mask per batch row (PR 31525's attention_mask, pads anywhere) on the
    fused shard-layout path: the mask rows are those of the attention batch entries (head
    group g of batch row bb is entry g*b + bb), so the result equals the relayout path's
    bit for bit (dQ within the gradient bar); one group is also compared with the
    oracle."""
    need_gpu()
    N, b, s, h, d, causal = case
    w = workloads.Workload("masked", 93, b=b, h=h, d=d, s=s, N=N, causal=causal, scale=1.0)
    ins = workloads.make_inputs(w, device="cuda")
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * w.index + 6)
    mask = torch.rand((b, s), generator=g) < 0.7
    mask[-1, s // 2:] = False          # a right-padded row: key blocks with no visible key
    res = []
    for fused in (False, True):
        step = UlyssesAttention(N, b, s, h, d, causal, key_mask=mask.to("cuda"), fused=fused)
        o = step.forward(ins["q"], ins["k"], ins["v"]).clone()
        lse = step.lse.clone()
        grads = [t.clone() for t in step.backward(ins["dout"])]
        torch.cuda.synchronize()
        check_status()
        res.append((o, lse, grads))
        del step
    (o0, l0, g0), (o1, l1, g1) = res
    assert torch.equal(o0.view(torch.int16), o1.view(torch.int16)), "out"
    assert torch.equal(l0, l1), "lse"
    for name, x, y in zip(("dk", "dv"), g0[1:], g1[1:]):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16)), name
    check_grad(f64(g1[0]), f64(g0[0]), "dq")
    # head group 0 against the oracle (its rows of the shard layout, regrouped by the oracle)
    orc = oracle.default()

    def group0(t):
        bits = t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        gr = orc.seq2head(bits, N, b, s, h, d)[0]
        return torch.from_numpy(gr.view(np.int16).copy()).view(torch.bfloat16).double().numpy()

    q, k, v, do = (group0(ins[n]) for n in ("q", "k", "v", "dout"))
    km = mask.numpy()
    ro, _ = orc.attn_fwd(q, k, v, causal, key_mask=km)
    rdq, rdk, rdv = orc.attn_bwd(q, k, v, do, causal, key_mask=km)
    check_out(group0(o1), ro, "group 0 out")
    check_grad(group0(g1[0]), rdq, "group 0 dq")
    check_grad(group0(g1[1]), rdk, "group 0 dk")
    check_grad(group0(g1[2]), rdv, "group 0 dv")


def test_fused_layout_needs_whole_tiles_per_shard():
    """Shards of 64 rows (the tiny workload) cannot be read as 128-row tiles: refused."""
    need_gpu()
    w = workloads.WORKLOADS["tiny"]
    ins = workloads.make_inputs(w, device="cuda")
    with pytest.raises(SpError) as e:
        sp_attn_fwd(ins["q"], ins["k"], ins["v"], True)
    assert e.value.code == 2          # SP_ERR_UNSUPPORTED
