"""The Ulysses attention step on one GPU, as a sequence of libsp calls.

forward  : Q/K/V shards --seq2head--> head groups --attn_fwd--> O groups --head2seq--> O shards
backward : dO shards --seq2head--> dO groups --attn_bwd--> dQ/dK/dV groups --head2seq--> shards

Shards are [N][b][s/N][h][d] and groups [N][b][s][h/N][d]; attention runs once over
all groups, viewed as N*b batch entries of h/N heads (heads are independent,
"Parallel multi-head attention" section 2).  Buffers are allocated once (torch) and
reused by every step.
"""
from __future__ import annotations

import contextlib

import torch

from .binding import (sp_attn_bwd, sp_attn_bwd_workspace_size, sp_attn_fwd, sp_attn_merge,
                      sp_relayout_head2seq, sp_relayout_seq2head)


class UlyssesAttention:
    def __init__(self, N: int, b: int, s: int, h: int, d: int, causal: bool = True,
                 key_len: torch.Tensor | None = None, softmax_scale: float | None = None,
                 device="cuda", timer=None, ring_chunks: int = 0,
                 key_mask: torch.Tensor | None = None):
        """`timer(name)`, if given, returns a context manager wrapped around each
        library call (used to bracket calls with CUDA events).  ring_chunks > 1 runs the
        attention blockwise over that many equal key chunks (ring attention) instead of
        in one call.  key_mask ([b][s] bool, True = key takes part) is a general key mask
        per batch row, applied in every head group."""
        if s % N or h % N:
            raise ValueError("s and h must be divisible by N")
        self.N, self.b, self.s, self.h, self.d = N, b, s, h, d
        self.causal = causal
        self.softmax_scale = softmax_scale
        self.timer = timer if timer is not None else (lambda name: contextlib.nullcontext())
        dev = torch.device(device)
        hl = h // N
        gshape = (N, b, s, hl, d)
        bf = dict(dtype=torch.bfloat16, device=dev)
        # key lengths per batch row, repeated for every head group (batch entry g*b + bb)
        self.key_len = None if key_len is None else key_len.to(dev, torch.int32).repeat(N)
        self.key_mask = None if key_mask is None else key_mask.to(dev).repeat(N, 1)
        self.qg, self.kg, self.vg = (torch.empty(gshape, **bf) for _ in range(3))
        self.og = torch.empty(gshape, **bf)
        self.dog = torch.empty(gshape, **bf)
        self.dqg, self.dkg, self.dvg = (torch.empty(gshape, **bf) for _ in range(3))
        self.lse = torch.empty((N * b, hl, s), dtype=torch.float32, device=dev)
        sshape = (N, b, s // N, h, d)
        self.o = torch.empty(sshape, **bf)
        self.dq, self.dk, self.dv = (torch.empty(sshape, **bf) for _ in range(3))
        ws = sp_attn_bwd_workspace_size(self._g(self.qg), self._g(self.kg), self._g(self.vg),
                                        causal, 0, self.key_len, softmax_scale)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.ring_chunks = int(ring_chunks)
        if self.ring_chunks > 1 and key_mask is not None:
            raise ValueError("ring attention here takes key_len, not a general key mask")
        if self.ring_chunks > 1:
            if s % self.ring_chunks:
                raise ValueError("s must be divisible by ring_chunks")
            c = s // self.ring_chunks
            self.chunks = [(n * c, (n + 1) * c) for n in range(self.ring_chunks)]
            self.ring_bufs = {}

    def _g(self, t: torch.Tensor) -> torch.Tensor:
        """Group buffer [N][b][s][hl][d] viewed as attention batch [N*b][s][hl][d]."""
        return t.view(self.N * self.b, self.s, self.h // self.N, self.d)

    def _to_groups(self, shards, groups, name):
        if self.N == 1:
            for x, y in zip(shards, groups):
                y.copy_(x)          # one shard is already the full sequence
            return
        with self.timer(name):
            sp_relayout_seq2head(list(shards), self.N, outs=list(groups))

    def _to_shards(self, groups, shards, name):
        if self.N == 1:
            for x, y in zip(groups, shards):
                y.copy_(x)
            return
        with self.timer(name):
            sp_relayout_head2seq(list(groups), self.N, outs=list(shards))

    def forward(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> torch.Tensor:
        """q, k, v: [N][b][s/N][h][d] shards -> O shards (same layout)."""
        self._to_groups((q, k, v), (self.qg, self.kg, self.vg), "seq2head_qkv")
        if self.ring_chunks > 1:
            out, lse, _ = ring_attention_fwd(self._g(self.qg), self._g(self.kg), self._g(self.vg),
                                             self.chunks, self.causal, 0, self.key_len,
                                             self.softmax_scale, bufs=self.ring_bufs,
                                             timer=self.timer)
            self.og = out.view(self.og.shape)
            self.lse = lse
        else:
            with self.timer("attn_fwd"):
                sp_attn_fwd(self._g(self.qg), self._g(self.kg), self._g(self.vg), self.causal,
                            0, self.key_len, self.softmax_scale, out=self._g(self.og),
                            lse=self.lse, key_mask=self.key_mask)
        self._to_shards((self.og,), (self.o,), "head2seq_o")
        return self.o

    def backward(self, dout: torch.Tensor):
        """dout shards -> (dq, dk, dv) shards; uses the last forward's O and lse."""
        self._to_groups((dout,), (self.dog,), "seq2head_do")
        if self.ring_chunks > 1:
            ring_attention_bwd(self._g(self.qg), self._g(self.kg), self._g(self.vg),
                               self._g(self.og), self.lse, self._g(self.dog), self.chunks,
                               self.causal, 0, self.key_len, self.softmax_scale,
                               dq=self._g(self.dqg), dk=self._g(self.dkg), dv=self._g(self.dvg),
                               workspace=self.workspace, timer=self.timer)
            self._to_shards((self.dqg, self.dkg, self.dvg), (self.dq, self.dk, self.dv),
                            "head2seq_grads")
            return self.dq, self.dk, self.dv
        with self.timer("attn_bwd"):
            sp_attn_bwd(self._g(self.qg), self._g(self.kg), self._g(self.vg), self._g(self.og),
                        self.lse, self._g(self.dog), self.causal, 0, self.key_len,
                        self.softmax_scale, dq=self._g(self.dqg), dk=self._g(self.dkg),
                        dv=self._g(self.dvg), workspace=self.workspace, key_mask=self.key_mask)
        self._to_shards((self.dqg, self.dkg, self.dvg), (self.dq, self.dk, self.dv),
                        "head2seq_grads")
        return self.dq, self.dk, self.dv


def _chunk_key_len(key_len, lo, hi):
    """Valid keys of the key chunk [lo, hi) for each batch entry (device int32)."""
    if key_len is None:
        return None
    return (key_len.to(torch.int32) - lo).clamp_(0, hi - lo).contiguous()


def ring_attention_fwd(q, k, v, chunks, causal=True, q_offset=0, key_len=None,
                       softmax_scale=None, bufs=None, timer=None):
    """Blockwise (ring) attention on one GPU: the keys are visited chunk by chunk, as the
    K/V blocks of a ring arrive at one device ("adv07: Sequence Parallel", sections 5
    and 7), and each chunk's (o, lse) is merged into an fp32 accumulator.

    q [B][sq][H][d], k/v [B][sk][H][d]; chunks = [(lo, hi), ...] partitioning [0, sk)
    in visiting order.  Returns (out bf16, lse fp32, o_acc fp32).  `bufs` (a dict, filled
    on first use) keeps the buffers between calls; `timer(name)` brackets each call."""
    B, sq, H, d = q.shape
    bufs = {} if bufs is None else bufs
    if "part" not in bufs:
        bufs["part"] = torch.empty((B, sq, H, d), dtype=torch.bfloat16, device=q.device)
        bufs["part_lse"] = torch.empty((B, H, sq), dtype=torch.float32, device=q.device)
        bufs["o_acc"] = torch.empty((B, sq, H, d), dtype=torch.float32, device=q.device)
        bufs["lse"] = torch.empty((B, H, sq), dtype=torch.float32, device=q.device)
        bufs["out"] = torch.empty((B, sq, H, d), dtype=torch.bfloat16, device=q.device)
    part, part_lse, o_acc, lse, out = (bufs[n] for n in ("part", "part_lse", "o_acc", "lse", "out"))
    timer = timer if timer is not None else (lambda name: contextlib.nullcontext())
    for n, (lo, hi) in enumerate(chunks):
        with timer("ring_chunk_fwd"):
            sp_attn_fwd(q, k[:, lo:hi], v[:, lo:hi], causal, q_offset,
                        _chunk_key_len(key_len, lo, hi), softmax_scale, out=part, lse=part_lse,
                        kv_offset=lo)
        with timer("ring_merge"):
            sp_attn_merge(part, part_lse, o_acc, lse, init=(n == 0),
                          o_out=out if n == len(chunks) - 1 else None)
    return out, lse, o_acc


def ring_attention_bwd(q, k, v, out, lse, dout, chunks, causal=True, q_offset=0, key_len=None,
                       softmax_scale=None, dq=None, dk=None, dv=None, workspace=None,
                       timer=None):
    """Backward of ring_attention_fwd, chunk by chunk with the merged out and lse: each
    chunk's call yields that chunk's dk, dv and adds its dq contribution to an fp32
    accumulator kept in the shared workspace."""
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws = workspace
    timer = timer if timer is not None else (lambda name: contextlib.nullcontext())
    for n, (lo, hi) in enumerate(chunks):
        kl = _chunk_key_len(key_len, lo, hi)
        if ws is None:
            size = sp_attn_bwd_workspace_size(q, k[:, lo:hi], v[:, lo:hi], causal, q_offset, kl,
                                              softmax_scale, kv_offset=lo)
            ws = torch.empty(max(size, 1), dtype=torch.uint8, device=q.device)
        with timer("ring_chunk_bwd"):
            sp_attn_bwd(q, k[:, lo:hi], v[:, lo:hi], out, lse, dout, causal, q_offset, kl,
                        softmax_scale, dq=dq, dk=dk[:, lo:hi], dv=dv[:, lo:hi], workspace=ws,
                        kv_offset=lo, dq_accumulate=(n > 0))
    return dq, dk, dv
