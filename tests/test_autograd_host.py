"""Host logic of the autograd entry points, on the CPU: with the library replaced by a
recorder that computes nothing, the calls that forward and backward make, their order and
their arguments (shapes, head groups, shard count, causal flag) are those of the Ulysses
step: regroup Q, K, V in one call, attend over N*b entries of h/N heads, regroup O; in the
backward regroup dO, run the attention backward, regroup dQ, dK, dV in one call."""
import ctypes

import pytest
import torch

import sequence_head_attention_seq_b300.binding as binding
from sequence_head_attention_seq_b300 import attention, seq_all_to_all, ulysses_attention


class _Recorder:
    """Stands in for libsp: records each call with the arguments that matter here."""

    def __init__(self):
        self.calls = []

    def __getattr__(self, name):
        if name.startswith("__"):
            raise AttributeError(name)
        rec = self

        def fn(*args):
            rec.calls.append((name, rec._summary(name, args)))
            return 64 if name == "sp_attn_bwd_workspace_size" else 0
        return fn

    @staticmethod
    def _summary(name, args):
        if name in ("sp_relayout_seq2head", "sp_relayout_head2seq"):
            return {"ntensors": args[2], "N": args[3], "b": args[4], "s": args[5], "h": args[6],
                    "d": args[7]}
        if name == "sp_relayout":
            shape = ctypes.cast(args[3], ctypes.POINTER(ctypes.c_int64))
            return {"N": args[2], "shape": tuple(shape[i] for i in range(4)),
                    "scatter": args[4], "gather": args[5]}
        if name.startswith("sp_attn"):
            p = args[0]._obj
            return {"B": p.B, "H": p.H, "sq": p.sq, "sk": p.sk, "d": p.d, "causal": p.causal,
                    "shards": p.seq_shards}
        return {}


@pytest.fixture
def rec(monkeypatch):
    r = _Recorder()
    monkeypatch.setattr(binding, "load", lambda build_if_missing=True: r)
    monkeypatch.setattr(binding, "_stream", lambda device: ctypes.c_void_p(0))

    def need_bf16(name, t):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.bfloat16:
            raise TypeError(name)
    monkeypatch.setattr(binding, "_need_bf16_cuda", need_bf16)
    return r


def _shards(N, b, s, h, d):
    return [torch.zeros((N, b, s // N, h, d), dtype=torch.bfloat16, requires_grad=True)
            for _ in range(3)]


def test_ulysses_attention_calls(rec):
    N, b, s, h, d = 4, 2, 512, 8, 64
    q, k, v = _shards(N, b, s, h, d)
    out = ulysses_attention(q, k, v, causal=True)
    assert out.shape == (N, b, s // N, h, d)
    group = {"B": N * b, "H": h // N, "sq": s, "sk": s, "d": d, "causal": 1, "shards": 1}
    regroup = {"N": N, "b": b, "s": s, "h": h, "d": d}
    assert rec.calls == [("sp_relayout_seq2head", {"ntensors": 3, **regroup}),
                         ("sp_attn_fwd", group),
                         ("sp_relayout_head2seq", {"ntensors": 1, **regroup})]
    rec.calls.clear()
    out.backward(torch.zeros_like(out))
    names = [c[0] for c in rec.calls]
    assert names == ["sp_relayout_seq2head", "sp_attn_bwd_workspace_size", "sp_attn_bwd",
                     "sp_relayout_head2seq"]
    assert rec.calls[0][1] == {"ntensors": 1, **regroup}
    assert rec.calls[2][1] == group
    assert rec.calls[3][1] == {"ntensors": 3, **regroup}
    assert q.grad.shape == q.shape and k.grad.shape == k.shape and v.grad.shape == v.shape


def test_ulysses_attention_fused_calls(rec):
    """fused=True: the kernels address the shard layout, so no regrouping call is made."""
    N, b, s, h, d = 2, 1, 256, 4, 128
    q, k, v = _shards(N, b, s, h, d)
    out = ulysses_attention(q, k, v, causal=False, fused=True)
    out.backward(torch.zeros_like(out))
    assert [c[0] for c in rec.calls] == ["sp_attn_fwd", "sp_attn_bwd_workspace_size",
                                         "sp_attn_bwd"]
    assert rec.calls[0][1] == {"B": N * b, "H": h // N, "sq": s, "sk": s, "d": d, "causal": 0,
                               "shards": N}


def test_one_shard_needs_no_regrouping(rec):
    q, k, v = _shards(1, 2, 128, 4, 64)
    out = ulysses_attention(q, k, v)
    assert out.shape == q.shape
    assert [c[0] for c in rec.calls] == ["sp_attn_fwd"]
    assert rec.calls[0][1]["B"] == 2 and rec.calls[0][1]["H"] == 4


def test_attention_saves_what_backward_needs(rec):
    B, sq, sk, H, d = 2, 100, 130, 3, 64
    q = torch.zeros((B, sq, H, d), dtype=torch.bfloat16, requires_grad=True)
    k = torch.zeros((B, sk, H, d), dtype=torch.bfloat16, requires_grad=True)
    v = torch.zeros((B, sk, H, d), dtype=torch.bfloat16, requires_grad=True)
    out = attention(q, k, v, causal=True, q_offset=30)
    out.backward(torch.zeros_like(out).transpose(0, 1).contiguous().transpose(0, 1))
    assert [c[0] for c in rec.calls] == ["sp_attn_fwd", "sp_attn_bwd_workspace_size",
                                         "sp_attn_bwd"]
    assert rec.calls[2][1] == {"B": B, "H": H, "sq": sq, "sk": sk, "d": d, "causal": 1,
                               "shards": 1}
    # no second-order gradients: differentiating the backward is refused
    out2 = attention(q, k, v)
    dout = torch.zeros_like(out2).requires_grad_()
    (g,) = torch.autograd.grad(out2, (q,), dout, create_graph=True)
    with pytest.raises(RuntimeError, match="differentiate twice"):
        g.sum().backward()


def test_seq_all_to_all_gradient_goes_the_other_way(rec):
    N, b, s, h, d = 4, 1, 64, 8, 16
    x = torch.zeros((N, b, s // N, h, d), dtype=torch.bfloat16, requires_grad=True)
    y = seq_all_to_all(x, N, 2, 1)
    assert y.shape == (N, b, s, h // N, d)
    y.backward(torch.zeros_like(y))
    assert rec.calls == [("sp_relayout", {"N": N, "shape": (b, s // N, h, d), "scatter": 2,
                                          "gather": 1}),
                         ("sp_relayout", {"N": N, "shape": (b, s, h // N, d), "scatter": 1,
                                          "gather": 2})]
    assert x.grad.shape == x.shape


# ---------------------------------------------------------------- the step class itself

def test_ulysses_step_calls(rec):
    """UlyssesAttention (the benchmark's step): the same six library calls per step,
    buffers reused from one step to the next."""
    from sequence_head_attention_seq_b300 import UlyssesAttention
    N, b, s, h, d = 2, 1, 256, 4, 128
    step = UlyssesAttention(N, b, s, h, d, causal=True, device="cpu")
    rec.calls.clear()
    shards = [torch.zeros((N, b, s // N, h, d), dtype=torch.bfloat16) for _ in range(4)]
    outs = []
    for _ in range(2):
        o = step.forward(*shards[:3])
        grads = step.backward(shards[3])
        outs.append((o.data_ptr(),) + tuple(g.data_ptr() for g in grads))
    names = [c[0] for c in rec.calls]
    one = ["sp_relayout_seq2head", "sp_attn_fwd", "sp_relayout_head2seq",
           "sp_relayout_seq2head", "sp_attn_bwd_workspace_size", "sp_attn_bwd",
           "sp_relayout_head2seq"]
    assert names == one + one
    assert outs[0] == outs[1]                  # the same output buffers every step
    group = {"B": N * b, "H": h // N, "sq": s, "sk": s, "d": d, "causal": 1, "shards": 1}
    assert rec.calls[1][1] == group and rec.calls[5][1] == group

