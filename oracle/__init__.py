"""Python face of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the product library
and its binding never do.  It shares no code with the CUDA path: it is built
from ``oracle.c`` alone with the host C compiler.

Every array the oracle sees is float64 (bf16 inputs are widened exactly by the
caller) except the relayout, which copies opaque 16-bit words.

What each function computes, and the page passage it follows, is stated in the
header of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_default = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("sq", ctypes.c_int),
        ("sk", ctypes.c_int), ("d", ctypes.c_int), ("causal", ctypes.c_int),
        ("q_offset", ctypes.c_int), ("key_len", ctypes.POINTER(ctypes.c_int32)),
        ("key_mask", ctypes.POINTER(ctypes.c_uint8)), ("scale", ctypes.c_double),
    ]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle source file with gcc (plain -O2, IEEE semantics kept)."""
    tmp = out + ".tmp%d" % os.getpid()
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Build _oracle.so from oracle.c when it is missing or older than the source."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            compile_source(_SRC, _LIB)
    return _LIB


def open_library(path: str):
    """Load a compiled oracle and declare its C signatures."""
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    pp = ctypes.POINTER(_Problem)
    u16 = ctypes.POINTER(ctypes.c_uint16)
    i = ctypes.c_int
    lib.oracle_attn_fwd.argtypes = [pp, dp, dp, dp, dp, dp]
    lib.oracle_attn_bwd.argtypes = [pp, dp, dp, dp, dp, dp, dp, dp]
    lib.oracle_attn_fwd_rows.argtypes = [pp, dp, dp, dp, i, i, i, i, dp, dp]
    lib.oracle_attn_bwd_rows.argtypes = [pp, dp, dp, dp, dp, i, i, i, i, dp, i, i, dp, dp]
    lib.oracle_seq2head.argtypes = [u16, u16, i, i, i, i, i]
    lib.oracle_head2seq.argtypes = [u16, u16, i, i, i, i, i]
    lib.oracle_attn_merge.argtypes = [i, i, i, i, i, dp, dp, dp, dp]
    lib.oracle_set_threads.argtypes = [i]
    for f in (lib.oracle_attn_fwd, lib.oracle_attn_bwd, lib.oracle_attn_fwd_rows,
              lib.oracle_attn_bwd_rows, lib.oracle_seq2head, lib.oracle_head2seq,
              lib.oracle_attn_merge,
              lib.oracle_set_threads, lib.oracle_get_threads):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _default
    if _default is None:
        path = build()
        with _lock:
            if _default is None:
                _default = open_library(path)
    return _default


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype.itemsize != 2:
        raise TypeError("relayout copies 16-bit words")
    return a.view(np.uint16)


class Problem:
    """Shapes and mask of one attention problem (q: [B][sq][H][d], k/v: [B][sk][H][d])."""

    def __init__(self, B, H, sq, sk, d, causal, q_offset=0, key_len=None, scale=None,
                 key_mask=None):
        self.B, self.H, self.sq, self.sk, self.d = int(B), int(H), int(sq), int(sk), int(d)
        self.causal = bool(causal)
        self.q_offset = int(q_offset)
        self.key_len = None if key_len is None else np.ascontiguousarray(
            np.asarray(key_len, dtype=np.int32))
        self.key_mask = None
        if key_mask is not None:
            m = np.ascontiguousarray(np.asarray(key_mask) != 0, dtype=np.uint8)
            if m.shape != (self.B, self.sk):
                raise ValueError("key_mask must be [B][sk]")
            self.key_mask = m
        self.scale = 1.0 / math.sqrt(d) if scale is None else float(scale)

    @classmethod
    def of(cls, q, k, causal, q_offset=0, key_len=None, scale=None, key_mask=None) -> "Problem":
        B, sq, H, d = q.shape
        return cls(B, H, sq, k.shape[1], d, causal, q_offset, key_len, scale, key_mask)

    def c_struct(self) -> _Problem:
        kl = (self.key_len.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
              if self.key_len is not None else ctypes.POINTER(ctypes.c_int32)())
        km = (self.key_mask.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8))
              if self.key_mask is not None else ctypes.POINTER(ctypes.c_uint8)())
        return _Problem(self.B, self.H, self.sq, self.sk, self.d, int(self.causal),
                        self.q_offset, kl, km, self.scale)


class Oracle:
    """Typed calls into one compiled oracle library (the default build, or a test's mutant)."""

    def __init__(self, lib):
        self.lib = lib

    def set_threads(self, n: int) -> None:
        """Thread count of the task pool (0 = all online cores)."""
        self.lib.oracle_set_threads(int(n))

    def threads(self) -> int:
        return int(self.lib.oracle_get_threads())

    def attn_fwd(self, q, k, v, causal, q_offset=0, key_len=None, scale=None, key_mask=None):
        """out [B][sq][H][d], lse [B][H][sq] (natural log) for all rows."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        P = Problem.of(q, k, causal, q_offset, key_len, scale, key_mask)
        out = np.empty_like(q)
        lse = np.empty((P.B, P.H, P.sq), dtype=np.float64)
        cp = P.c_struct()
        if self.lib.oracle_attn_fwd(ctypes.byref(cp), _ptr(q), _ptr(k), _ptr(v), _ptr(out),
                                    _ptr(lse)):
            raise ValueError("oracle_attn_fwd rejected the problem")
        return out, lse

    def attn_bwd(self, q, k, v, dout, causal, q_offset=0, key_len=None, scale=None,
                 key_mask=None):
        """dq [B][sq][H][d], dk/dv [B][sk][H][d] for all rows."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        P = Problem.of(q, k, causal, q_offset, key_len, scale, key_mask)
        dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
        cp = P.c_struct()
        if self.lib.oracle_attn_bwd(ctypes.byref(cp), _ptr(q), _ptr(k), _ptr(v), _ptr(dout),
                                    _ptr(dq), _ptr(dk), _ptr(dv)):
            raise ValueError("oracle_attn_bwd rejected the problem")
        return dq, dk, dv

    def attn_fwd_rows(self, q, k, v, b, h, i0, i1, causal, q_offset=0, key_len=None,
                      scale=None, key_mask=None):
        """out [i1-i0][d], lse [i1-i0] for query rows [i0, i1) of head (b, h)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        P = Problem.of(q, k, causal, q_offset, key_len, scale, key_mask)
        out = np.empty((max(i1 - i0, 0) + 1, P.d), dtype=np.float64)
        lse = np.empty((max(i1 - i0, 0) + 1,), dtype=np.float64)
        cp = P.c_struct()
        if self.lib.oracle_attn_fwd_rows(ctypes.byref(cp), _ptr(q), _ptr(k), _ptr(v), b, h,
                                         i0, i1, _ptr(out), _ptr(lse)):
            raise ValueError("oracle_attn_fwd_rows rejected the request")
        return out[: i1 - i0], lse[: i1 - i0]

    def attn_bwd_rows(self, q, k, v, dout, b, h, i0, i1, j0, j1, causal, q_offset=0,
                      key_len=None, scale=None, key_mask=None):
        """dq rows [i0, i1) and dk/dv rows [j0, j1) of head (b, h)."""
        q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
        P = Problem.of(q, k, causal, q_offset, key_len, scale, key_mask)
        dq = np.zeros((max(i1 - i0, 0) + 1, P.d), dtype=np.float64)
        dk = np.zeros((max(j1 - j0, 0) + 1, P.d), dtype=np.float64)
        dv = np.zeros((max(j1 - j0, 0) + 1, P.d), dtype=np.float64)
        cp = P.c_struct()
        if self.lib.oracle_attn_bwd_rows(ctypes.byref(cp), _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(dout), b, h, i0, i1, _ptr(dq), j0, j1,
                                         _ptr(dk), _ptr(dv)):
            raise ValueError("oracle_attn_bwd_rows rejected the request")
        return dq[: i1 - i0], dk[: j1 - j0], dv[: j1 - j0]

    def attn_merge(self, outs, lses):
        """Combine per-key-chunk results: outs[k] [B][sq][H][d], lses[k] [B][H][sq] ->
        (out, lse) of attention over the union of the chunks' keys."""
        outs = np.ascontiguousarray(np.stack([_f64(o) for o in outs]))
        lses = np.ascontiguousarray(np.stack([_f64(l) for l in lses]))
        n, B, sq, H, d = outs.shape
        out = np.empty((B, sq, H, d), dtype=np.float64)
        lse = np.empty((B, H, sq), dtype=np.float64)
        if self.lib.oracle_attn_merge(B, H, sq, d, n, _ptr(outs), _ptr(lses), _ptr(out),
                                      _ptr(lse)):
            raise ValueError("oracle_attn_merge rejected the request")
        return out, lse

    def seq2head(self, x, N, b, s, h, d) -> np.ndarray:
        """[N][b][s/N][h][d] -> [N][b][s][h/N][d], as opaque 16-bit words."""
        x = _u16(x)
        out = np.empty((N, b, s, h // N, d), dtype=np.uint16)
        if self.lib.oracle_seq2head(x.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                    N, b, s, h, d):
            raise ValueError("oracle_seq2head: s and h must divide by N")
        return out

    def head2seq(self, x, N, b, s, h, d) -> np.ndarray:
        """[N][b][s][h/N][d] -> [N][b][s/N][h][d], as opaque 16-bit words."""
        x = _u16(x)
        out = np.empty((N, b, s // N, h, d), dtype=np.uint16)
        if self.lib.oracle_head2seq(x.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                    out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                    N, b, s, h, d):
            raise ValueError("oracle_head2seq: s and h must divide by N")
        return out


# ---------------------------------------------------------------- projections and layer
#
# "Parallel multi-head attention", sections 2.1-2.3 and 3.1-3.2: the input is projected by
# ColumnParallelLinear wq, wk, wv (nn.Linear, y = x W^T with W [out][in]), attention runs
# per head, and the concatenated heads are projected by a RowParallelLinear wo.  On one
# device the weights are whole; wq, wk, wv are stacked into one [3*h*d][dim] weight, so
# the projection's output is the packed [..][3][h][d] layout.  Matrix products are
# numpy's (a library primitive); the regrouping is the seq->head index formula written
# with reshape/transpose.


def linear_fwd(x, w):
    """y = x W^T (fp64)."""
    return _f64(x) @ _f64(w).T


def linear_bwd(dy, x, w):
    """(dx, dW) of y = x W^T: dx = dy W, dW = dy^T x (fp64, over all leading dims of x)."""
    dy, x, w = _f64(dy), _f64(x), _f64(w)
    dy2 = dy.reshape(-1, dy.shape[-1])
    x2 = x.reshape(-1, x.shape[-1])
    return (dy2 @ w).reshape(x.shape[:-1] + (w.shape[1],)), dy2.T @ x2


def _groups_of(t, N):
    """[N][b][s/N][h][d] shards -> [N][b][s][h/N][d] head groups (fp64)."""
    n, b, sl, h, d = t.shape
    full = t.transpose(1, 0, 2, 3, 4).reshape(b, n * sl, h, d)
    return full.reshape(b, n * sl, N, h // N, d).transpose(2, 0, 1, 3, 4)


def _shards_of(g, N):
    """[N][b][s][h/N][d] head groups -> [N][b][s/N][h][d] shards (fp64)."""
    n, b, s, hl, d = g.shape
    full = g.transpose(1, 2, 0, 3, 4).reshape(b, s, n * hl, d)
    return full.reshape(b, N, s // N, n * hl, d).transpose(1, 0, 2, 3, 4)


class Layer:
    """The attention layer of the sequence-parallel step on shards x [N][b][s/N][dim]:
    qkv = x Wqkv^T, Ulysses regrouping, causal attention per head, regrouping back,
    out = O Wo^T.  Weights: wqkv [3*h*d][dim], wo [dim][h*d]."""

    def __init__(self, orc, N, h, d, causal=True):
        self.orc, self.N, self.h, self.d, self.causal = orc, N, h, d, causal

    def forward(self, x, wqkv, wo):
        N, h, d = self.N, self.h, self.d
        x = _f64(x)
        n, b, sl, dim = x.shape
        qkv = linear_fwd(x, wqkv).reshape(n, b, sl, 3, h, d)
        groups = [_groups_of(qkv[:, :, :, t], N) for t in range(3)]     # [N][b][s][hl][d]
        o_groups = np.empty_like(groups[0])
        for g in range(N):
            o_groups[g], _ = self.orc.attn_fwd(groups[0][g], groups[1][g], groups[2][g],
                                               self.causal)
        o = _shards_of(o_groups, N).reshape(n, b, sl, h * d)
        self.saved = (x, wqkv, wo, groups, o)
        return linear_fwd(o, wo)

    def backward(self, dout):
        """(dx, dwqkv, dwo) for the last forward."""
        N, h, d = self.N, self.h, self.d
        x, wqkv, wo, groups, o = self.saved
        n, b, sl, _ = x.shape
        do, dwo = linear_bwd(dout, o, wo)
        do_groups = _groups_of(do.reshape(n, b, sl, h, d), N)
        grads = [np.empty_like(groups[0]) for _ in range(3)]
        for g in range(N):
            dq, dk, dv = self.orc.attn_bwd(groups[0][g], groups[1][g], groups[2][g],
                                           do_groups[g], self.causal)
            grads[0][g], grads[1][g], grads[2][g] = dq, dk, dv
        dqkv = np.stack([_shards_of(t, N) for t in grads], axis=3).reshape(n, b, sl, 3 * h * d)
        dx, dwqkv = linear_bwd(dqkv, x, wqkv)
        return dx, dwqkv, dwo


def default() -> Oracle:
    """The oracle built from oracle.c in this directory."""
    return Oracle(_load())


def __getattr__(name):
    # module-level shortcuts: oracle.attn_fwd(...), oracle.seq2head(...), ...
    if name in ("set_threads", "threads", "attn_fwd", "attn_bwd", "attn_fwd_rows",
                "attn_bwd_rows", "attn_merge", "seq2head", "head2seq"):
        return getattr(default(), name)
    raise AttributeError(name)
