"""Thin ctypes binding of libsp (include/sp.h), same names as the C ABI.

Only argument marshalling happens here: tensor checks, strides, data
pointers and the current CUDA stream.  Every step of the computation runs in
libsp's kernels.  PyTorch provides device memory and streams.

If libsp.so cannot be loaded (or built), every call raises ``SpError``: there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None

SP_OK = 0
STATUS_NAMES = {0: "SP_OK", 1: "SP_ERR_INVALID_ARG", 2: "SP_ERR_UNSUPPORTED",
                3: "SP_ERR_MISALIGNED", 4: "SP_ERR_CUDA", 5: "SP_ERR_TIMEOUT",
                6: "SP_ERR_WORKSPACE"}
MAX_RELAYOUT_TENSORS = 8

# Every symbol include/sp.h declares.
EXPORTS = ["sp_relayout_seq2head", "sp_relayout_head2seq", "sp_relayout", "sp_relayout_seq2head_packed",
           "sp_relayout_head2seq_packed", "sp_attn_fwd",
           "sp_attn_bwd_workspace_size", "sp_attn_bwd", "sp_attn_merge", "sp_linear_fwd",
           "sp_linear_bwd", "sp_attn_bwd_noalloc", "sp_ulysses_host_workspace_size",
           "sp_ulysses_step_host", "sp_selftest_wait_timeout",
           "sp_get_device_status", "sp_status_string"]
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024   # SP_NOALLOC_SCRATCH_BYTES


class SpError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = int(code)
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)}")


class SpAttnParams(ctypes.Structure):
    """Mirror of sp_attn_params."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("q_stride", ctypes.c_int64 * 3), ("k_stride", ctypes.c_int64 * 3),
        ("v_stride", ctypes.c_int64 * 3), ("o_stride", ctypes.c_int64 * 3),
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("sq", ctypes.c_int), ("sk", ctypes.c_int),
        ("d", ctypes.c_int), ("causal", ctypes.c_int), ("q_offset", ctypes.c_int),
        ("kv_offset", ctypes.c_int),
        ("key_len", ctypes.c_void_p), ("softmax_scale", ctypes.c_float),
        ("dq_accumulate", ctypes.c_int),
        ("key_mask", ctypes.c_void_p), ("key_mask_stride", ctypes.c_int64),
        ("seq_shards", ctypes.c_int),
    ]


class SpMergeParams(ctypes.Structure):
    """Mirror of sp_merge_params."""
    _fields_ = [
        ("B", ctypes.c_int), ("H", ctypes.c_int), ("sq", ctypes.c_int), ("d", ctypes.c_int),
        ("init", ctypes.c_int),
        ("o_part", ctypes.c_void_p), ("part_stride", ctypes.c_int64 * 3),
        ("lse_part", ctypes.c_void_p), ("o_acc", ctypes.c_void_p), ("lse_acc", ctypes.c_void_p),
        ("o_out", ctypes.c_void_p), ("out_stride", ctypes.c_int64 * 3),
    ]


class SpUlyssesHostParams(ctypes.Structure):
    """Mirror of sp_ulysses_host_params."""
    _fields_ = [
        ("N", ctypes.c_int), ("b", ctypes.c_int), ("s", ctypes.c_int), ("h", ctypes.c_int),
        ("d", ctypes.c_int), ("causal", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("key_len", ctypes.c_void_p),
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("dout", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p),
        ("dv", ctypes.c_void_p),
    ]


def library_path() -> str:
    return os.path.join(_PKG, "libsp.so")


def load(build_if_missing: bool = True):
    """Load libsp.so (building it with nvcc first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        from . import build as _build
        try:
            if build_if_missing and _build.stale():
                _build.build()
        except Exception as e:  # noqa: BLE001 - report why the native library is unavailable
            raise RuntimeError(f"libsp could not be built: {e}") from e
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libsp.so not found at {path}")
        lib = ctypes.CDLL(path)
        vpp = ctypes.POINTER(ctypes.c_void_p)
        i = ctypes.c_int
        for name in ("sp_relayout_seq2head", "sp_relayout_head2seq"):
            f = getattr(lib, name)
            f.argtypes = [vpp, vpp, i, i, i, i, i, i, ctypes.c_void_p]
            f.restype = i
        lib.sp_relayout.argtypes = [ctypes.c_void_p, ctypes.c_void_p, i,
                                    ctypes.POINTER(ctypes.c_int64), i, i, ctypes.c_void_p]
        lib.sp_relayout.restype = i
        lib.sp_relayout_seq2head_packed.argtypes = [ctypes.c_void_p, vpp, i, i, i, i, i,
                                                    ctypes.c_void_p]
        lib.sp_relayout_seq2head_packed.restype = i
        lib.sp_relayout_head2seq_packed.argtypes = [vpp, ctypes.c_void_p, i, i, i, i, i,
                                                    ctypes.c_void_p]
        lib.sp_relayout_head2seq_packed.restype = i
        pp = ctypes.POINTER(SpAttnParams)
        lib.sp_attn_fwd.argtypes = [pp, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        lib.sp_attn_fwd.restype = i
        lib.sp_attn_bwd_workspace_size.argtypes = [pp]
        lib.sp_attn_bwd_workspace_size.restype = ctypes.c_size_t
        lib.sp_attn_bwd.argtypes = [pp] + [ctypes.c_void_p] * 7 + [ctypes.c_size_t, ctypes.c_void_p]
        lib.sp_attn_bwd.restype = i
        lib.sp_attn_bwd_noalloc.argtypes = [pp] + [ctypes.c_void_p] * 7
        lib.sp_attn_bwd_noalloc.restype = i
        lib.sp_attn_merge.argtypes = [ctypes.POINTER(SpMergeParams), ctypes.c_void_p]
        lib.sp_attn_merge.restype = i
        vp = ctypes.c_void_p
        lib.sp_linear_fwd.argtypes = [vp, vp, vp, i, i, i, vp]
        lib.sp_linear_fwd.restype = i
        lib.sp_linear_bwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
        lib.sp_linear_bwd.restype = i
        lib.sp_ulysses_host_workspace_size.argtypes = [i, i, i, i, i, i]
        lib.sp_ulysses_host_workspace_size.restype = ctypes.c_size_t
        lib.sp_ulysses_step_host.argtypes = [ctypes.POINTER(SpUlyssesHostParams), vp,
                                             ctypes.c_size_t, vp, vp, vp]
        lib.sp_ulysses_step_host.restype = i
        lib.sp_selftest_wait_timeout.argtypes = [ctypes.c_void_p]
        lib.sp_selftest_wait_timeout.restype = i
        lib.sp_get_device_status.argtypes = [ctypes.c_void_p]
        lib.sp_get_device_status.restype = i
        lib.sp_status_string.argtypes = [i]
        lib.sp_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check(fn: str, rc: int) -> None:
    if rc != SP_OK:
        raise SpError(fn, rc)


def _need_bf16_cuda(name: str, t: torch.Tensor) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _ptr_array(ts):
    arr = (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])
    return ctypes.cast(arr, ctypes.POINTER(ctypes.c_void_p)), arr


def _relayout(fn_name: str, inputs, N: int, b: int, s: int, h: int, d: int, out_shape, outs):
    lib = load()
    if not 1 <= len(inputs) <= MAX_RELAYOUT_TENSORS:
        raise ValueError("relayout moves 1..8 tensors per call")
    for n, t in enumerate(inputs):
        _need_bf16_cuda(f"in[{n}]", t)
        if not t.is_contiguous():
            raise ValueError("relayout inputs must be contiguous")
    if outs is None:
        outs = [torch.empty(out_shape, dtype=torch.bfloat16, device=inputs[0].device)
                for _ in inputs]
    for n, t in enumerate(outs):
        _need_bf16_cuda(f"out[{n}]", t)
        if not t.is_contiguous() or t.numel() != math.prod(out_shape):
            raise ValueError("relayout outputs must be contiguous with the output size")
    pin, keep_in = _ptr_array(inputs)
    pout, keep_out = _ptr_array(outs)
    rc = getattr(lib, fn_name)(pin, pout, len(inputs), N, b, s, h, d, _stream(inputs[0].device))
    _check(fn_name, rc)
    return outs


def sp_relayout_seq2head(inputs, N: int, outs=None):
    """Sequence shards [N][b][s/N][h][d] -> head groups [N][b][s][h/N][d] (one launch)."""
    x = inputs[0]
    if x.dim() != 5 or x.shape[0] != N:
        raise ValueError("expected [N][b][s/N][h][d] shard tensors")
    _, b, sl, h, d = x.shape
    if h % N:
        raise ValueError("h must be divisible by N")
    return _relayout("sp_relayout_seq2head", inputs, N, b, sl * N, h, d,
                     (N, b, sl * N, h // N, d), outs)


def sp_relayout_head2seq(inputs, N: int, outs=None):
    """Head groups [N][b][s][h/N][d] -> sequence shards [N][b][s/N][h][d] (one launch)."""
    x = inputs[0]
    if x.dim() != 5 or x.shape[0] != N:
        raise ValueError("expected [N][b][s][h/N][d] group tensors")
    _, b, s, hl, d = x.shape
    if s % N:
        raise ValueError("s must be divisible by N")
    return _relayout("sp_relayout_head2seq", inputs, N, b, s, hl * N, d,
                     (N, b, s // N, hl * N, d), outs)


def sp_relayout(x, N: int, scatter_dim: int, gather_dim: int, out=None):
    """The all-to-all in scatter/gather form on N stacked per-rank tensors [N][b][x][y][d]:
    (2, 1) is sequence shards -> head groups, (1, 2) head groups -> sequence shards."""
    lib = load()
    _need_bf16_cuda("x", x)
    if x.dim() != 5 or x.shape[0] != N or not x.is_contiguous():
        raise ValueError("expected N contiguous per-rank tensors [N][b][x][y][d]")
    _, b, xd, yd, d = x.shape
    if (scatter_dim, gather_dim) == (2, 1):
        oshape = (N, b, xd * N, yd // N, d)
    elif (scatter_dim, gather_dim) == (1, 2):
        oshape = (N, b, xd // N, yd * N, d)
    else:
        oshape = tuple(x.shape)
    if out is None:
        out = torch.empty(oshape, dtype=x.dtype, device=x.device)
    shape = (ctypes.c_int64 * 4)(b, xd, yd, d)
    rc = lib.sp_relayout(x.data_ptr(), out.data_ptr(), N, shape, scatter_dim, gather_dim,
                         _stream(x.device))
    _check("sp_relayout", rc)
    return out


def _same_layout(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Equal strides on every dimension longer than 1 (others are never stepped)."""
    return all(n == 1 or sa == sb for n, sa, sb in zip(a.shape, a.stride(), b.stride()))


def _strides(t: torch.Tensor, name: str):
    if t.dim() != 4:
        raise ValueError(f"{name} must be [B][S][H][d]")
    if t.stride(3) != 1:
        raise ValueError(f"{name}: head_dim must be contiguous")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def _mask_rows(key_mask, B: int, sk: int):
    """key_mask as device bytes in rows of a 16-byte-multiple stride (padded copy if needed)."""
    if not isinstance(key_mask, torch.Tensor) or not key_mask.is_cuda:
        raise ValueError("key_mask must be a CUDA tensor")
    if tuple(key_mask.shape) != (B, sk):
        raise ValueError(f"key_mask must be [B][sk] = [{B}][{sk}]")
    m = key_mask.to(torch.uint8) if key_mask.dtype == torch.bool else key_mask
    if m.dtype != torch.uint8:
        raise ValueError("key_mask must be bool or uint8")
    ok = (m.stride(1) == 1 and m.stride(0) % 16 == 0 and m.stride(0) >= sk
          and m.data_ptr() % 16 == 0)
    if not ok:
        stride = (sk + 15) // 16 * 16
        padded = torch.zeros((B, max(stride, 16)), dtype=torch.uint8, device=m.device)
        padded[:, :sk] = m
        m = padded
    return m


def attn_dims(q):
    """(B, sq, H, d, N) of a query tensor: [B][sq][H][d] (N = 1) or, in the sequence-shard
    layout [N][b][s/N][N*H][d], B = N*b batch entries (entry g*b + bb = head group g of
    batch row bb) over the full sequence sq = s."""
    if q.dim() == 5:
        N, b, sl, h, d = q.shape
        if h % N:
            raise ValueError("shard tensors need a head count divisible by N")
        return N * b, N * sl, h // N, d, N
    B, sq, H, d = q.shape
    return B, sq, H, d, 1


def make_params(q, k, v, o_like, causal: bool, q_offset: int = 0, key_len=None,
                softmax_scale=None, kv_offset: int = 0, key_mask=None) -> SpAttnParams:
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_bf16_cuda(name, t)
    p = SpAttnParams()
    p.q, p.k, p.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
    B, sq, H, d, N = attn_dims(q)
    if N > 1:
        # sequence-shard layout: all tensors [N][b][s/N][N*H][d], contiguous
        for name, t in (("k", k), ("v", v), ("o", o_like)):
            if t.shape != q.shape:
                raise ValueError(f"{name} must have the shard shape of q")
        for name, t in (("q", q), ("k", k), ("v", v), ("o", o_like)):
            if not t.is_contiguous():
                raise ValueError(f"{name}: shard tensors must be contiguous")
        zero = (ctypes.c_int64 * 3)(0, 0, 0)
        p.q_stride = p.k_stride = p.v_stride = p.o_stride = zero
        sk = sq
    else:
        if k.shape[0] != B or k.shape[2] != H or k.shape[3] != d or v.shape != k.shape:
            raise ValueError("k and v must be [B][sk][H][d] matching q")
        p.q_stride = _strides(q, "q")
        p.k_stride = _strides(k, "k")
        p.v_stride = _strides(v, "v")
        p.o_stride = _strides(o_like, "o")
        sk = k.shape[1]
    p.seq_shards = N
    p.B, p.H, p.sq, p.sk, p.d = B, H, sq, sk, d
    p.causal = 1 if causal else 0
    p.q_offset = int(q_offset)
    p.kv_offset = int(kv_offset)
    if key_len is not None:
        if key_len.dtype != torch.int32 or not key_len.is_cuda or key_len.numel() != B:
            raise ValueError("key_len must be a CUDA int32 tensor of B entries")
        p.key_len = key_len.data_ptr()
    else:
        p.key_len = None
    p.softmax_scale = float(softmax_scale) if softmax_scale is not None else 0.0
    if key_mask is not None:
        m = _mask_rows(key_mask, B, sk)
        p.key_mask = m.data_ptr()
        p.key_mask_stride = m.stride(0)
        p._keep = m                     # keeps a padded copy alive while p is in use
    else:
        p.key_mask = None
        p.key_mask_stride = 0
    return p


def sp_relayout_seq2head_packed(qkv, N: int, outs=None):
    """Packed sequence shards [N][b][s/N][3][h][d] -> Q, K, V head groups
    [N][b][s][h/N][d] (one launch)."""
    lib = load()
    _need_bf16_cuda("qkv", qkv)
    if qkv.dim() != 6 or qkv.shape[0] != N or qkv.shape[3] != 3 or not qkv.is_contiguous():
        raise ValueError("qkv must be contiguous [N][b][s/N][3][h][d]")
    _, b, sl, _, h, d = qkv.shape
    s = N * sl
    shape = (N, b, s, h // N, d)
    if outs is None:
        outs = [torch.empty(shape, dtype=torch.bfloat16, device=qkv.device) for _ in range(3)]
    for n, t in enumerate(outs):
        _need_bf16_cuda(f"out[{n}]", t)
        if not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"outputs must be contiguous {shape}")
    pout, keep = _ptr_array(outs)
    rc = lib.sp_relayout_seq2head_packed(qkv.data_ptr(), pout, N, b, s, h, d,
                                         _stream(qkv.device))
    _check("sp_relayout_seq2head_packed", rc)
    return outs


def sp_relayout_head2seq_packed(groups, N: int, out=None):
    """Three head-group tensors [N][b][s][h/N][d] -> packed shards [N][b][s/N][3][h][d]."""
    lib = load()
    if len(groups) != 3:
        raise ValueError("three head-group tensors")
    for n, t in enumerate(groups):
        _need_bf16_cuda(f"in[{n}]", t)
        if not t.is_contiguous() or t.shape != groups[0].shape or t.dim() != 5:
            raise ValueError("inputs must be contiguous [N][b][s][h/N][d] of one shape")
    _, b, s, hl, d = groups[0].shape
    h = hl * N
    shape = (N, b, s // N, 3, h, d)
    if out is None:
        out = torch.empty(shape, dtype=torch.bfloat16, device=groups[0].device)
    _need_bf16_cuda("out", out)
    if not out.is_contiguous() or tuple(out.shape) != shape:
        raise ValueError(f"out must be contiguous {shape}")
    pin, keep = _ptr_array(list(groups))
    rc = lib.sp_relayout_head2seq_packed(pin, out.data_ptr(), N, b, s, h, d,
                                         _stream(out.device))
    _check("sp_relayout_head2seq_packed", rc)
    return out


def sp_attn_fwd(q, k, v, causal: bool = True, q_offset: int = 0, key_len=None,
                softmax_scale=None, out=None, lse=None, kv_offset: int = 0, key_mask=None):
    """out (bf16, layout of q) and lse [B][H][sq] fp32 (natural log).  q, k, v are
    [B][sq][H][d] / [B][sk][H][d], or all three [N][b][s/N][N*H][d] sequence shards (the
    Ulysses regrouping is then done by the kernels' own addressing)."""
    lib = load()
    B, sq, H, d, _ = attn_dims(q)
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    if lse is None:
        lse = torch.empty((B, H, sq), dtype=torch.float32, device=q.device)
    _need_bf16_cuda("out", out)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or lse.shape != (B, H, sq):
        raise ValueError("lse must be contiguous fp32 [B][H][sq]")
    p = make_params(q, k, v, out, causal, q_offset, key_len, softmax_scale, kv_offset, key_mask)
    rc = lib.sp_attn_fwd(ctypes.byref(p), out.data_ptr(), lse.data_ptr(), _stream(q.device))
    _check("sp_attn_fwd", rc)
    return out, lse


def sp_attn_bwd_workspace_size(q, k, v, causal: bool = True, q_offset: int = 0, key_len=None,
                               softmax_scale=None, kv_offset: int = 0, key_mask=None) -> int:
    lib = load()
    p = make_params(q, k, v, q, causal, q_offset, key_len, softmax_scale, kv_offset, key_mask)
    return int(lib.sp_attn_bwd_workspace_size(ctypes.byref(p)))


def sp_attn_bwd(q, k, v, out, lse, dout, causal: bool = True, q_offset: int = 0, key_len=None,
                softmax_scale=None, dq=None, dk=None, dv=None, workspace=None,
                kv_offset: int = 0, dq_accumulate: bool = False, key_mask=None):
    """dq, dk, dv (bf16, layouts of q, k, v) from the forward's out/lse and dout.

    Ring / blockwise attention: call once per key chunk (k, v of the chunk, its
    kv_offset, the merged out/lse), with dq_accumulate=True after the first chunk and
    the same workspace each time; dq then holds the sum over the chunks so far."""
    lib = load()
    _need_bf16_cuda("out", out)
    _need_bf16_cuda("dout", dout)
    if out.shape != dout.shape or not _same_layout(out, dout):
        raise ValueError("out and dout must share shape and strides")
    p = make_params(q, k, v, out, causal, q_offset, key_len, softmax_scale, kv_offset, key_mask)
    p.dq_accumulate = 1 if dq_accumulate else 0

    def like(t):
        return torch.empty_strided(t.size(), t.stride(), dtype=t.dtype, device=t.device)

    dq = like(q) if dq is None else dq
    dk = like(k) if dk is None else dk
    dv = like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _need_bf16_cuda(name, t)
        if t.shape != ref.shape or not _same_layout(t, ref):
            raise ValueError(f"{name} must have the shape and strides of its input")
    need = int(lib.sp_attn_bwd_workspace_size(ctypes.byref(p)))
    if workspace is None:
        if dq_accumulate:
            raise ValueError("dq_accumulate needs the workspace of the previous call")
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    rc = lib.sp_attn_bwd(ctypes.byref(p), out.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                         dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), _stream(q.device))
    _check("sp_attn_bwd", rc)
    return dq, dk, dv


def sp_attn_bwd_noalloc(q, k, v, out, lse, dout, causal: bool = True, q_offset: int = 0,
                        key_len=None, softmax_scale=None, dq=None, dk=None, dv=None,
                        kv_offset: int = 0, key_mask=None):
    """sp_attn_bwd with the library's own fixed device scratch instead of a workspace.

    For callers that must not allocate device memory during the call: the C entry
    point allocates nothing (pass preallocated dq/dk/dv to keep this wrapper from
    allocating them either).  Problems needing more than NOALLOC_SCRATCH_BYTES of
    workspace raise SpError(SP_ERR_WORKSPACE); concurrent calls on unordered
    streams share the scratch and must not overlap.
    """
    lib = load()
    _need_bf16_cuda("out", out)
    _need_bf16_cuda("dout", dout)
    if out.shape != dout.shape or not _same_layout(out, dout):
        raise ValueError("out and dout must share shape and strides")
    p = make_params(q, k, v, out, causal, q_offset, key_len, softmax_scale, kv_offset, key_mask)

    def like(t):
        return torch.empty_strided(t.size(), t.stride(), dtype=t.dtype, device=t.device)

    dq = like(q) if dq is None else dq
    dk = like(k) if dk is None else dk
    dv = like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        _need_bf16_cuda(name, t)
        if t.shape != ref.shape or not _same_layout(t, ref):
            raise ValueError(f"{name} must have the shape and strides of its input")
    rc = lib.sp_attn_bwd_noalloc(ctypes.byref(p), out.data_ptr(), lse.data_ptr(),
                                 dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                 _stream(q.device))
    _check("sp_attn_bwd_noalloc", rc)
    return dq, dk, dv


def sp_attn_merge(o_part, lse_part, o_acc, lse_acc, init: bool, o_out=None):
    """Merge one key chunk's (o_part bf16 [B][sq][H][d], lse_part fp32 [B][H][sq]) into
    the running (o_acc fp32 [B][sq][H][d], lse_acc fp32 [B][H][sq]) in place; init starts a
    new accumulation; o_out (bf16, layout of o_part) also receives the merged output."""
    lib = load()
    _need_bf16_cuda("o_part", o_part)
    B, sq, H, d = o_part.shape
    for name, t, shape in (("lse_part", lse_part, (B, H, sq)), ("o_acc", o_acc, (B, sq, H, d)),
                           ("lse_acc", lse_acc, (B, H, sq))):
        if (t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous()
                or tuple(t.shape) != shape):
            raise ValueError(f"{name} must be contiguous CUDA fp32 of shape {shape}")
    p = SpMergeParams()
    p.B, p.H, p.sq, p.d = B, H, sq, d
    p.init = 1 if init else 0
    p.o_part = o_part.data_ptr()
    p.part_stride = _strides(o_part, "o_part")
    p.lse_part = lse_part.data_ptr()
    p.o_acc = o_acc.data_ptr()
    p.lse_acc = lse_acc.data_ptr()
    if o_out is not None:
        _need_bf16_cuda("o_out", o_out)
        if o_out.shape != o_part.shape:
            raise ValueError("o_out must have the shape of o_part")
        p.o_out = o_out.data_ptr()
        p.out_stride = _strides(o_out, "o_out")
    else:
        p.o_out = None
    rc = lib.sp_attn_merge(ctypes.byref(p), _stream(o_part.device))
    _check("sp_attn_merge", rc)
    return o_acc, lse_acc


def _rows(t: torch.Tensor, name: str, width: int):
    """A contiguous bf16 CUDA tensor viewed as rows of `width` elements."""
    _need_bf16_cuda(name, t)
    if not t.is_contiguous() or t.shape[-1] != width:
        raise ValueError(f"{name} must be contiguous with last dimension {width}")
    return t.numel() // width


def sp_linear_fwd(x, w, out=None):
    """y = x W^T for W [out_features][in_features]; x [..., in] -> y [..., out]."""
    lib = load()
    n_out, n_in = w.shape
    M = _rows(x, "x", n_in)
    _rows(w, "w", n_in)
    if out is None:
        out = torch.empty((*x.shape[:-1], n_out), dtype=torch.bfloat16, device=x.device)
    if _rows(out, "out", n_out) != M:
        raise ValueError("out must hold one row per row of x")
    rc = lib.sp_linear_fwd(x.data_ptr(), w.data_ptr(), out.data_ptr(), M, n_in, n_out,
                           _stream(x.device))
    _check("sp_linear_fwd", rc)
    return out


def sp_linear_bwd(dy, x, w, dx=None, dw=None, accumulate_dw: bool = False,
                  need_dx: bool = True):
    """dx = dy W and dW = dy^T x (or dW += dy^T x) for y = x W^T."""
    lib = load()
    n_out, n_in = w.shape
    M = _rows(x, "x", n_in)
    if _rows(dy, "dy", n_out) != M:
        raise ValueError("dy must hold one row per row of x")
    if need_dx and dx is None:
        dx = torch.empty_like(x)
    if dw is None:
        if accumulate_dw:
            raise ValueError("accumulate_dw needs the dw to add to")
        dw = torch.empty_like(w)
    if dx is not None and _rows(dx, "dx", n_in) != M:
        raise ValueError("dx must have the shape of x")
    _rows(dw, "dw", n_in)
    rc = lib.sp_linear_bwd(dy.data_ptr(), x.data_ptr(), w.data_ptr(),
                           dx.data_ptr() if dx is not None else None, dw.data_ptr(), M, n_in,
                           n_out, 1 if accumulate_dw else 0, _stream(x.device))
    _check("sp_linear_bwd", rc)
    return dx, dw


def sp_ulysses_host_workspace_size(N: int, b: int, s: int, h: int, d: int,
                                   causal: bool) -> int:
    return int(load().sp_ulysses_host_workspace_size(N, b, s, h, d, 1 if causal else 0))


def sp_ulysses_step_host(q, k, v, dout, o, dq, dk, dv, N: int, causal: bool, workspace,
                         h2d_stream, d2h_stream, key_len=None, softmax_scale: float = 0.0):
    """One Ulysses step on page-locked HOST shards [N, b, s/N, h, d] (bf16): o, dq, dk, dv
    receive the results.  The kernels run on the current stream of the workspace's
    device, the transfers on h2d_stream and d2h_stream (torch.cuda.Stream)."""
    lib = load()
    Nn, b, sl, h, d = q.shape
    if Nn != N:
        raise ValueError(f"q has {Nn} shards, N = {N}")
    for name, t in (("q", q), ("k", k), ("v", v), ("dout", dout), ("o", o), ("dq", dq),
                    ("dk", dk), ("dv", dv)):
        if (t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous()
                or tuple(t.shape) != (N, b, sl, h, d)):
            raise ValueError(f"{name} must be a contiguous host bf16 tensor of shape "
                             f"{(N, b, sl, h, d)}")
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise ValueError("workspace must be a CUDA uint8 tensor")
    p = SpUlyssesHostParams()
    p.N, p.b, p.s, p.h, p.d = N, b, sl * N, h, d
    p.causal = 1 if causal else 0
    p.softmax_scale = float(softmax_scale)
    if key_len is not None:
        if key_len.dtype != torch.int32 or not key_len.is_cuda or key_len.numel() != b:
            raise ValueError("key_len must be a CUDA int32 tensor of b entries")
        p.key_len = key_len.data_ptr()
    else:
        p.key_len = None
    p.q, p.k, p.v, p.dout = q.data_ptr(), k.data_ptr(), v.data_ptr(), dout.data_ptr()
    p.o, p.dq, p.dk, p.dv = o.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    rc = lib.sp_ulysses_step_host(ctypes.byref(p), workspace.data_ptr(), workspace.numel(),
                                  _stream(workspace.device), h2d_stream.cuda_stream,
                                  d2h_stream.cuda_stream)
    _check("sp_ulysses_step_host", rc)
    return o, dq, dk, dv


def sp_selftest_wait_timeout(device=None) -> None:
    """Enqueue the wait-timeout self-test on the current stream (see include/sp.h)."""
    _check("sp_selftest_wait_timeout", load().sp_selftest_wait_timeout(_stream(device)))


def sp_get_device_status(device=None) -> int:
    """Synchronise the current stream and return (and clear) the kernels' status code."""
    lib = load()
    return int(lib.sp_get_device_status(_stream(device)))


def sp_status_string(code: int) -> str:
    return load().sp_status_string(int(code)).decode()
