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
                      sp_linear_bwd, sp_linear_fwd, sp_relayout_head2seq,
                      sp_relayout_head2seq_packed, sp_relayout_seq2head,
                      sp_relayout_seq2head_packed, sp_ulysses_host_workspace_size,
                      sp_ulysses_step_host)


class UlyssesAttention:
    def __init__(self, N: int, b: int, s: int, h: int, d: int, causal: bool = True,
                 key_len: torch.Tensor | None = None, softmax_scale: float | None = None,
                 device="cuda", timer=None, ring_chunks: int = 0,
                 key_mask: torch.Tensor | None = None, fused: bool = False):
        """`timer(name)`, if given, returns a context manager wrapped around each
        library call (used to bracket calls with CUDA events).  ring_chunks > 1 runs the
        attention blockwise over that many equal key chunks (ring attention) instead of
        in one call.  key_mask ([b][s] bool, True = key takes part) is a general key mask
        per batch row, applied in every head group.  fused=True lets the attention kernels
        read and write the sequence shards directly (the regrouping is done by their own
        addressing) instead of running the two relayouts; N == 1 needs no regrouping."""
        if s % N or h % N:
            raise ValueError("s and h must be divisible by N")
        if fused and ring_chunks > 1:
            raise ValueError("ring attention runs on the head-group layout (fused=False)")
        if ring_chunks > 1 and key_mask is not None:
            raise ValueError("ring attention here takes key_len, not a general key mask")
        self.N, self.b, self.s, self.h, self.d = N, b, s, h, d
        self.causal = causal
        self.softmax_scale = softmax_scale
        self.timer = timer if timer is not None else (lambda name: contextlib.nullcontext())
        self.direct = fused or N == 1          # attention straight on the shard tensors
        dev = torch.device(device)
        hl = h // N
        bf = dict(dtype=torch.bfloat16, device=dev)
        # key lengths / mask per batch row, repeated for every head group (entry g*b + bb)
        self.key_len = None if key_len is None else key_len.to(dev, torch.int32).repeat(N)
        self.key_mask = None if key_mask is None else key_mask.to(dev).repeat(N, 1)
        self.lse = torch.empty((N * b, hl, s), dtype=torch.float32, device=dev)
        sshape = (N, b, s // N, h, d)
        self.o = torch.empty(sshape, **bf)
        self.dq, self.dk, self.dv = (torch.empty(sshape, **bf) for _ in range(3))
        if not self.direct:
            gshape = (N, b, s, hl, d)
            self.qg, self.kg, self.vg = (torch.empty(gshape, **bf) for _ in range(3))
            self.og = torch.empty(gshape, **bf)
            self.dog = torch.empty(gshape, **bf)
            self.dqg, self.dkg, self.dvg = (torch.empty(gshape, **bf) for _ in range(3))
            like = self._g(self.qg)
        else:
            like = self._a(self.o)
        ws = sp_attn_bwd_workspace_size(like, like, like, causal, 0, self.key_len, softmax_scale)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)
        self.ring_chunks = int(ring_chunks)
        if self.ring_chunks > 1:
            if s % self.ring_chunks:
                raise ValueError("s must be divisible by ring_chunks")
            c = s // self.ring_chunks
            self.chunks = [(n * c, (n + 1) * c) for n in range(self.ring_chunks)]
            self.ring_bufs = {}

    def _g(self, t: torch.Tensor) -> torch.Tensor:
        """Group buffer [N][b][s][hl][d] viewed as attention batch [N*b][s][hl][d]."""
        return t.view(self.N * self.b, self.s, self.h // self.N, self.d)

    def _a(self, t: torch.Tensor) -> torch.Tensor:
        """A shard tensor as the attention kernels take it directly: [b][s][h][d] for one
        shard, else the shard layout itself."""
        return t.view(self.b, self.s, self.h, self.d) if self.N == 1 else t

    def _to_groups(self, shards, groups, name):
        with self.timer(name):
            sp_relayout_seq2head(list(shards), self.N, outs=list(groups))

    def _to_shards(self, groups, shards, name):
        with self.timer(name):
            sp_relayout_head2seq(list(groups), self.N, outs=list(shards))

    def _attention_inputs(self):
        if self.direct:
            return self._a(self._q), self._a(self._k), self._a(self._v)
        return self._g(self.qg), self._g(self.kg), self._g(self.vg)

    def forward(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor) -> torch.Tensor:
        """q, k, v: [N][b][s/N][h][d] shards -> O shards (same layout)."""
        self._q, self._k, self._v = q, k, v
        if not self.direct:
            self._to_groups((q, k, v), (self.qg, self.kg, self.vg), "seq2head_qkv")
        aq, ak, av = self._attention_inputs()
        if self.ring_chunks > 1:
            out, lse, _ = ring_attention_fwd(aq, ak, av, self.chunks, self.causal, 0,
                                             self.key_len, self.softmax_scale,
                                             bufs=self.ring_bufs, timer=self.timer)
            if self.direct:
                self.o.copy_(out.view(self.o.shape))
            else:
                self.og = out.view(self.og.shape)
            self.lse = lse
        else:
            out = self._a(self.o) if self.direct else self._g(self.og)
            with self.timer("attn_fwd"):
                sp_attn_fwd(aq, ak, av, self.causal, 0, self.key_len, self.softmax_scale,
                            out=out, lse=self.lse, key_mask=self.key_mask)
        if not self.direct:
            self._to_shards((self.og,), (self.o,), "head2seq_o")
        return self.o

    def backward(self, dout: torch.Tensor):
        """dout shards -> (dq, dk, dv) shards; uses the last forward's inputs, O and lse."""
        aq, ak, av = self._attention_inputs()
        if self.direct:
            ao, ado = self._a(self.o), self._a(dout)
            grads = (self._a(self.dq), self._a(self.dk), self._a(self.dv))
        else:
            self._to_groups((dout,), (self.dog,), "seq2head_do")
            ao, ado = self._g(self.og), self._g(self.dog)
            grads = (self._g(self.dqg), self._g(self.dkg), self._g(self.dvg))
        if self.ring_chunks > 1:
            ring_attention_bwd(aq, ak, av, ao, self.lse, ado, self.chunks, self.causal, 0,
                               self.key_len, self.softmax_scale, dq=grads[0], dk=grads[1],
                               dv=grads[2], workspace=self.workspace, timer=self.timer)
        else:
            with self.timer("attn_bwd"):
                sp_attn_bwd(aq, ak, av, ao, self.lse, ado, self.causal, 0, self.key_len,
                            self.softmax_scale, dq=grads[0], dk=grads[1], dv=grads[2],
                            workspace=self.workspace, key_mask=self.key_mask)
        if not self.direct:
            self._to_shards((self.dqg, self.dkg, self.dvg), (self.dq, self.dk, self.dv),
                            "head2seq_grads")
        return self.dq, self.dk, self.dv


class UlyssesHostStep:
    """The Ulysses step of UlyssesAttention on page-locked HOST shards [N, b, s/N, h, d]:
    step() moves the inputs in, runs forward and backward and moves o, dq, dk, dv out,
    with each head group's transfers overlapping another group's kernels (the copy
    engines regroup sequence shards into head groups on the way).  Owns the device
    workspace and the two transfer streams; the kernels run on the current stream."""

    def __init__(self, N, b, s, h, d, causal=True, key_len=None, softmax_scale=0.0,
                 device=None):
        device = torch.device(device) if device is not None else torch.device("cuda")
        self.N, self.causal = N, causal
        self.softmax_scale = softmax_scale or 0.0
        # valid keys per batch row, on the device (the same for every head group)
        self.key_len = (None if key_len is None
                        else key_len.to(device, torch.int32).contiguous())
        nbytes = sp_ulysses_host_workspace_size(N, b, s, h, d, causal)
        if nbytes == 0:
            raise ValueError("unsupported host-step geometry")
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        self.h2d = torch.cuda.Stream(device)
        self.d2h = torch.cuda.Stream(device)

    def step(self, q, k, v, dout, o, dq, dk, dv):
        return sp_ulysses_step_host(q, k, v, dout, o, dq, dk, dv, self.N, self.causal,
                                    self.workspace, self.h2d, self.d2h, key_len=self.key_len,
                                    softmax_scale=self.softmax_scale)


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


class AttentionLayer:
    """The attention layer of the sequence-parallel step ("Parallel multi-head attention",
    sections 2-3: ColumnParallel q/k/v projections, attention per head, RowParallel
    output projection) on sequence shards x [N][b][s/N][dim]:

        qkv = x Wqkv^T          one GEMM into the packed [N][b][s/N][3][h][d] layout
        Q, K, V groups          sp_relayout_seq2head_packed (one launch)
        O groups                sp_attn_fwd
        O shards                sp_relayout_head2seq
        out = O Wo^T            one GEMM

    and the backward back to dx, dWqkv, dWo.  wqkv [3*h*d][dim], wo [dim][h*d] (bf16)."""

    def __init__(self, N: int, b: int, s: int, h: int, d: int, dim: int, causal: bool = True,
                 device="cuda", timer=None):
        if s % N or h % N:
            raise ValueError("s and h must be divisible by N")
        self.N, self.b, self.s, self.h, self.d, self.dim = N, b, s, h, d, dim
        self.causal = causal
        self.timer = timer if timer is not None else (lambda name: contextlib.nullcontext())
        dev = torch.device(device)
        bf = dict(dtype=torch.bfloat16, device=dev)
        sl, hl = s // N, h // N
        self.qkv = torch.empty((N, b, sl, 3, h, d), **bf)
        self.groups = [torch.empty((N, b, s, hl, d), **bf) for _ in range(3)]
        self.og = torch.empty((N, b, s, hl, d), **bf)
        self.o = torch.empty((N, b, sl, h, d), **bf)
        self.out = torch.empty((N, b, sl, dim), **bf)
        self.lse = torch.empty((N * b, hl, s), dtype=torch.float32, device=dev)
        self.do = torch.empty((N, b, sl, h, d), **bf)
        self.dog = torch.empty((N, b, s, hl, d), **bf)
        self.dgroups = [torch.empty((N, b, s, hl, d), **bf) for _ in range(3)]
        self.dqkv = torch.empty((N, b, sl, 3, h, d), **bf)
        self.dx = torch.empty((N, b, sl, dim), **bf)
        self.dwqkv = torch.empty((3 * h * d, dim), **bf)
        self.dwo = torch.empty((dim, h * d), **bf)
        g = self._g(self.og)
        ws = sp_attn_bwd_workspace_size(g, g, g, causal)
        self.workspace = torch.empty(max(ws, 1), dtype=torch.uint8, device=dev)

    def _g(self, t):
        return t.view(self.N * self.b, self.s, self.h // self.N, self.d)

    def forward(self, x, wqkv, wo):
        self._x, self._wqkv, self._wo = x, wqkv, wo
        with self.timer("proj_qkv"):
            sp_linear_fwd(x, wqkv, out=self.qkv.view(*x.shape[:-1], -1))
        with self.timer("seq2head_qkv"):
            sp_relayout_seq2head_packed(self.qkv, self.N, outs=self.groups)
        with self.timer("attn_fwd"):
            sp_attn_fwd(*(self._g(t) for t in self.groups), self.causal, out=self._g(self.og),
                        lse=self.lse)
        with self.timer("head2seq_o"):
            sp_relayout_head2seq([self.og], self.N, outs=[self.o])
        with self.timer("proj_o"):
            sp_linear_fwd(self.o.view(*self.o.shape[:3], -1), wo, out=self.out)
        return self.out

    def backward(self, dout):
        """-> (dx, dwqkv, dwo) for the last forward."""
        o2 = self.o.view(*self.o.shape[:3], -1)
        with self.timer("proj_o_bwd"):
            sp_linear_bwd(dout, o2, self._wo, dx=self.do.view(o2.shape), dw=self.dwo)
        with self.timer("seq2head_do"):
            sp_relayout_seq2head([self.do], self.N, outs=[self.dog])
        with self.timer("attn_bwd"):
            sp_attn_bwd(*(self._g(t) for t in self.groups), self._g(self.og), self.lse,
                        self._g(self.dog), self.causal, dq=self._g(self.dgroups[0]),
                        dk=self._g(self.dgroups[1]), dv=self._g(self.dgroups[2]),
                        workspace=self.workspace)
        with self.timer("head2seq_grads"):
            sp_relayout_head2seq_packed(self.dgroups, self.N, out=self.dqkv)
        with self.timer("proj_qkv_bwd"):
            sp_linear_bwd(self.dqkv.view(*self._x.shape[:-1], -1), self._x, self._wqkv,
                          dx=self.dx, dw=self.dwqkv)
        return self.dx, self.dwqkv, self.dwo
