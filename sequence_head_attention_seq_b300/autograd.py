"""The library's calls as torch.autograd Functions, so that attention and the Ulysses
regrouping sit inside a model's autograd graph.

This is how the pages' systems use the path: the sequence-parallel attention of
transformers PR 31525 ("Support deepspeed sequence parallel") and of the
long-context-attention issue wraps an all-to-all (sequence shards -> head groups), the
local attention and the inverse all-to-all, and its backward runs the same three steps in
reverse (the all-to-all of the gradients goes the other way).  Every step runs in libsp;
these Functions only route tensors and keep what the backward needs (q, k, v, out and the
per-row log-sum-exp).  The backward passes are not themselves differentiable (no
second-order gradients).

    attention(q, k, v, ...)            softmax(q k^T * scale + mask) v, [B][s][H][d] tensors
                                       or [N][b][s/N][N*H][d] sequence shards
    seq_all_to_all(x, N, scatter, gather)
                                       one tensor's regrouping; its gradient is the inverse
    ulysses_attention(q, k, v, ...)    shards -> head groups -> attention -> shards, with
                                       Q, K, V (and dQ, dK, dV) moved in one launch each
"""
from __future__ import annotations

import torch
from torch.autograd.function import once_differentiable

from .binding import (sp_attn_bwd, sp_attn_fwd, sp_relayout, sp_relayout_head2seq,
                      sp_relayout_seq2head)


class _Attention(torch.autograd.Function):
    """out = attention(q, k, v); backward through sp_attn_bwd with the saved out and lse."""

    @staticmethod
    def forward(ctx, q, k, v, causal, q_offset, key_len, softmax_scale, key_mask):
        o, lse = sp_attn_fwd(q, k, v, causal, q_offset, key_len, softmax_scale,
                             key_mask=key_mask)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.args = (causal, q_offset, key_len, softmax_scale, key_mask)
        return o

    @staticmethod
    @once_differentiable
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        causal, q_offset, key_len, softmax_scale, key_mask = ctx.args
        # the library takes dout with the strides of out, which it allocated contiguous
        do = do.contiguous()
        dq, dk, dv = sp_attn_bwd(q, k, v, o, lse, do, causal, q_offset, key_len,
                                 softmax_scale, key_mask=key_mask)
        return dq, dk, dv, None, None, None, None, None


def attention(q, k, v, causal: bool = True, q_offset: int = 0, key_len=None,
              softmax_scale=None, key_mask=None) -> torch.Tensor:
    """Attention with autograd ("adv07: Sequence Parallel", section 3 Q4: out[i] =
    softmax(q[i] K^T / sqrt(d)) V over the keys j <= q_offset + i when causal).

    q [B][sq][H][d], k and v [B][sk][H][d] (any strides with d contiguous), or all three
    in the sequence-shard layout [N][b][s/N][N*H][d], in which case the kernels do the
    regrouping by their own addressing and out comes back in the shard layout (key_len
    then has N*b entries, entry g*b + bb for head group g of batch row bb; s/N must be a
    multiple of 128).  key_len: optional CUDA int32 [B]; key_mask: optional CUDA bool or
    uint8 [B][sk].  Gradients flow to q, k and v."""
    return _Attention.apply(q, k, v, causal, q_offset, key_len, softmax_scale, key_mask)


class _SeqAllToAll(torch.autograd.Function):
    """One tensor's all-to-all in scatter/gather form; the gradient takes the inverse."""

    @staticmethod
    def forward(ctx, x, N, scatter_dim, gather_dim):
        ctx.args = (N, scatter_dim, gather_dim)
        return sp_relayout(x.contiguous(), N, scatter_dim, gather_dim)

    @staticmethod
    @once_differentiable
    def backward(ctx, g):
        N, scatter_dim, gather_dim = ctx.args
        return sp_relayout(g.contiguous(), N, gather_dim, scatter_dim), None, None, None


def seq_all_to_all(x, N: int, scatter_dim: int, gather_dim: int) -> torch.Tensor:
    """The sequence-parallel all-to-all of transformers PR 31525 on N stacked per-rank
    tensors [N][b][x][y][d] with autograd: (scatter 2, gather 1) regroups sequence shards
    into head groups, (1, 2) the reverse."""
    return _SeqAllToAll.apply(x, N, scatter_dim, gather_dim)


def _full_grads(grads, shapes):
    """Gradients of every output, contiguous, with zeros for outputs that received none."""
    ref = next(g for g in grads if g is not None)
    return [g.contiguous() if g is not None else
            torch.zeros(shapes[n], dtype=ref.dtype, device=ref.device)
            for n, g in enumerate(grads)]


class _ShardsToGroups(torch.autograd.Function):
    """Several shard tensors [N][b][s/N][h][d] -> head groups [N][b][s][h/N][d] in one
    launch; the backward regroups their gradients back in one launch."""

    @staticmethod
    def forward(ctx, N, *shards):
        ctx.N = N
        outs = sp_relayout_seq2head([t.contiguous() for t in shards], N)
        ctx.shapes = [o.shape for o in outs]
        return tuple(outs)

    @staticmethod
    @once_differentiable
    def backward(ctx, *grads):
        return (None, *sp_relayout_head2seq(_full_grads(grads, ctx.shapes), ctx.N))


class _GroupsToShards(torch.autograd.Function):
    """Head groups -> sequence shards in one launch; the backward goes the other way."""

    @staticmethod
    def forward(ctx, N, *groups):
        ctx.N = N
        outs = sp_relayout_head2seq([t.contiguous() for t in groups], N)
        ctx.shapes = [o.shape for o in outs]
        return tuple(outs)

    @staticmethod
    @once_differentiable
    def backward(ctx, *grads):
        return (None, *sp_relayout_seq2head(_full_grads(grads, ctx.shapes), ctx.N))


def ulysses_attention(q, k, v, causal: bool = True, key_len=None, softmax_scale=None,
                      key_mask=None, fused: bool = False) -> torch.Tensor:
    """The Ulysses attention step with autograd on sequence shards q, k, v
    [N][b][s/N][h][d] (shard r = sequence rows [r*s/N, (r+1)*s/N) of every head, as the
    PR 31525 data collator splits them): regroup into N head groups of h/N heads over the
    full sequence, attend, regroup the output back into shards.  key_len ([b] int32) and
    key_mask ([b][s]) are per batch row and apply to every head group.

    fused=True lets the attention kernels read and write the shard layout directly
    instead of running the two regroupings (needs s/N to be a multiple of 128)."""
    if q.dim() != 5:
        raise ValueError("expected sequence shards [N][b][s/N][h][d]")
    N, b, sl, h, d = q.shape
    if h % N:
        raise ValueError("h must be divisible by N")
    s, hl = sl * N, h // N
    kl = None if key_len is None else key_len.to(q.device, torch.int32).repeat(N)
    km = None if key_mask is None else key_mask.to(q.device).repeat(N, 1)
    if fused or N == 1:
        if N == 1:
            view = (b, s, h, d)
            out = attention(q.reshape(view), k.reshape(view), v.reshape(view), causal, 0, kl,
                            softmax_scale, km)
            return out.view(q.shape)
        return attention(q, k, v, causal, 0, kl, softmax_scale, km)
    qg, kg, vg = _ShardsToGroups.apply(N, q, k, v)
    gview = (N * b, s, hl, d)
    og = attention(qg.view(gview), kg.view(gview), vg.view(gview), causal, 0, kl,
                   softmax_scale, km)
    (o,) = _GroupsToShards.apply(N, og.view(N, b, s, hl, d))
    return o
