"""The Ulysses step on host-resident shards (sp_ulysses_step_host): the copy engines
regroup each head group between the host shard layout and a head-major device buffer
while they move it, and every group runs as its own attention problem.  Each group's
kernels do the same arithmetic in the same order as the one launch over all groups of
the device step, so o, dk and dv are identical bit for bit, and dq (whose fp32
additions happen in any order) agrees within the gradient bar; one small step is also
checked group by group against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import check_grad, check_out, check_status, f64, need_gpu
from sequence_head_attention_seq_b300 import (SpError, UlyssesAttention, UlyssesHostStep,
                                              workloads)

pytestmark = pytest.mark.gpu

SHAPES = [
    # b = 2: the copies go shard by shard and row by row of the batch
    workloads.Workload("host_shards2", 92, b=2, h=4, d=64, s=512, N=2, causal=True, scale=1.0),
    # padded keys, non-causal, d = 128
    workloads.Workload("host_shards4_pad", 93, b=2, h=8, d=128, s=2048, N=4, causal=False,
                       scale=1.0, key_len_range=(700, 2048)),
    # b = 1: one 2-D copy per tensor and head group
    workloads.WORKLOADS["llama7b"],
    # one shard: the single head group goes as two halves of its heads
    workloads.Workload("host_one_shard", 95, b=1, h=4, d=128, s=384, N=1, causal=True,
                       scale=1.0),
    # one head per group: no group can be split
    workloads.Workload("host_one_head", 96, b=1, h=2, d=64, s=512, N=2, causal=True, scale=1.0),
]


def _pinned(t):
    return t.cpu().pin_memory()


def _host_step(w, ins):
    host_in = [_pinned(ins[n]) for n in ("q", "k", "v", "dout")]
    host_out = [torch.empty_like(host_in[0]).pin_memory() for _ in range(4)]
    step = UlyssesHostStep(w.N, w.b, w.s, w.h, w.d, w.causal, key_len=ins["key_len"])
    step.step(*host_in, *host_out)
    torch.cuda.synchronize()
    check_status()
    return host_out


@pytest.mark.parametrize("w", SHAPES, ids=[w.name for w in SHAPES])
def test_host_step_equals_device_step(w):
    need_gpu()
    ins = workloads.make_inputs(w, device="cuda")
    dev = UlyssesAttention(w.N, w.b, w.s, w.h, w.d, w.causal, key_len=ins["key_len"])
    o = dev.forward(ins["q"], ins["k"], ins["v"]).cpu()
    dq, dk, dv = (t.cpu() for t in dev.backward(ins["dout"]))
    torch.cuda.synchronize()
    check_status()
    ho, hdq, hdk, hdv = _host_step(w, ins)
    for name, a, b in (("o", o, ho), ("dk", dk, hdk), ("dv", dv, hdv)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), name
    check_grad(f64(hdq), f64(dq), "dq")


def test_host_step_against_oracle():
    need_gpu()
    w = SHAPES[0]
    ins = workloads.make_inputs(w, device="cuda")
    o, dq, dk, dv = _host_step(w, ins)
    orc = oracle.default()

    def groups(t):
        bits = t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)
        g = orc.seq2head(bits, w.N, w.b, w.s, w.h, w.d)
        return torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16).double().numpy()

    q, k, v, do = (groups(ins[n]) for n in ("q", "k", "v", "dout"))
    og, dqg, dkg, dvg = (groups(t) for t in (o, dq, dk, dv))
    for g in range(w.N):
        ro, _ = orc.attn_fwd(q[g], k[g], v[g], w.causal)
        rdq, rdk, rdv = orc.attn_bwd(q[g], k[g], v[g], do[g], w.causal)
        check_out(og[g], ro, f"group {g} out")
        check_grad(dqg[g], rdq, f"group {g} dq")
        check_grad(dkg[g], rdk, f"group {g} dk")
        check_grad(dvg[g], rdv, f"group {g} dv")


def test_host_step_refuses_pageable_memory():
    """Host buffers must be page-locked (the copies could not overlap otherwise)."""
    need_gpu()
    w = SHAPES[0]
    ins = workloads.make_inputs(w, device="cuda")
    host_in = [ins[n].cpu() for n in ("q", "k", "v", "dout")]
    host_out = [torch.empty_like(host_in[0]) for _ in range(4)]
    step = UlyssesHostStep(w.N, w.b, w.s, w.h, w.d, w.causal)
    with pytest.raises(SpError) as e:
        step.step(*host_in, *host_out)
    assert e.value.code == 1          # SP_ERR_INVALID_ARG
