"""Host-only checks of the C ABI: the library builds and loads without a GPU,
exports exactly what include/sp.h declares, and rejects bad arguments before
launching anything (fake, never-dereferenced pointers are enough for that)."""
import ctypes
import os
import re
import subprocess

import pytest

from sequence_head_attention_seq_b300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sp.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, CUDA, TIMEOUT, WORKSPACE = range(7)
FAKE = 0x10000          # 16-byte aligned, never dereferenced
FAKE_ODD = 0x10008      # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sp_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_binding_exports():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(sp_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(lib, name)


def test_build_targets_sm_103a_only():
    from sequence_head_attention_seq_b300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_status_strings(lib):
    for code in range(7):
        assert binding.sp_status_string(code)
    assert binding.sp_status_string(99) == "unknown status"


def _arr(*vals):
    a = (ctypes.c_void_p * len(vals))(*vals)
    return ctypes.cast(a, ctypes.POINTER(ctypes.c_void_p)), a


@pytest.mark.parametrize("fn", ["sp_relayout_seq2head", "sp_relayout_head2seq"])
def test_relayout_validation(lib, fn):
    f = getattr(lib, fn)
    pin, a = _arr(FAKE, FAKE)
    pout, b = _arr(FAKE * 2, FAKE * 3)
    assert f(pin, pout, 2, 0, 1, 8, 4, 64, None) == INVALID          # N < 1
    assert f(pin, pout, 2, 3, 1, 8, 3, 64, None) == INVALID          # s % N
    assert f(pin, pout, 2, 2, 1, 8, 3, 64, None) == INVALID          # h % N
    assert f(pin, pout, 0, 2, 1, 8, 4, 64, None) == INVALID          # ntensors
    assert f(pin, pout, 9, 2, 1, 8, 4, 64, None) == INVALID
    assert f(None, pout, 2, 2, 1, 8, 4, 64, None) == INVALID
    pnull, c = _arr(FAKE, 0)
    assert f(pnull, pout, 2, 2, 1, 8, 4, 64, None) == INVALID
    podd, e = _arr(FAKE, FAKE_ODD)
    assert f(podd, pout, 2, 2, 1, 8, 4, 64, None) == MISALIGNED


def _params(**kw):
    p = binding.SpAttnParams()
    p.q = p.k = p.v = FAKE
    for name in ("q_stride", "k_stride", "v_stride", "o_stride"):
        setattr(p, name, (ctypes.c_int64 * 3)(128 * 256 * 4, 128 * 4, 128))
    p.B, p.H, p.sq, p.sk, p.d = 1, 4, 256, 256, 128
    p.causal, p.q_offset = 1, 0
    p.key_len = None
    p.softmax_scale = 0.0
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), UNSUPPORTED),
    (dict(d=256), UNSUPPORTED),
    (dict(causal=2), INVALID),
    (dict(q_offset=-1), INVALID),
    (dict(kv_offset=-1), INVALID),
    (dict(dq_accumulate=2), INVALID),
    (dict(key_mask=FAKE_ODD, key_mask_stride=256), MISALIGNED),
    (dict(key_mask=FAKE, key_mask_stride=264), MISALIGNED),     # stride not a multiple of 16
    (dict(key_mask=FAKE, key_mask_stride=240), INVALID),        # stride < sk
    (dict(seq_shards=-1), INVALID),
    (dict(seq_shards=3), INVALID),                              # B = 1 not a multiple of 3
    (dict(seq_shards=2, B=2, sk=512), INVALID),                 # shard layout needs sq == sk
    (dict(seq_shards=4, B=4), UNSUPPORTED),                     # 256 / 4 = 64-row shards
    (dict(kv_offset=(1 << 30) - 100), UNSUPPORTED),   # kv_offset + sk above 2^30
    (dict(sq=-1), INVALID),
    (dict(B=-2), INVALID),
    (dict(q=None), INVALID),
    (dict(k=None), INVALID),                          # keys exist: k and v are required
    (dict(v=None), INVALID),
    (dict(k=FAKE_ODD), MISALIGNED),
    (dict(q_stride=(ctypes.c_int64 * 3)(4, 4, 4)), MISALIGNED),
    (dict(key_len=FAKE + 2), MISALIGNED),
])
def test_attn_validation(lib, kw, code):
    p = _params(**kw)
    assert lib.sp_attn_fwd(ctypes.byref(p), FAKE, FAKE, None) == code
    assert lib.sp_attn_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                           1 << 40, None) == code
    assert lib.sp_attn_bwd_workspace_size(ctypes.byref(p)) == 0


def test_null_pointers_for_tensors_without_elements(lib):
    """A tensor with no elements may be NULL (PyTorch gives empty tensors no storage):
    here the problems are empty, so the calls return before anything is launched."""
    p = _params(sq=0, q=None)
    assert lib.sp_attn_fwd(ctypes.byref(p), None, None, None) == OK
    p = _params(B=0, q=None, k=None, v=None)
    assert lib.sp_attn_fwd(ctypes.byref(p), None, None, None) == OK
    assert lib.sp_attn_bwd(ctypes.byref(p), None, None, None, None, None, None, FAKE, 1 << 20,
                           None) == OK
    # a problem with query rows still needs its outputs
    p = _params(sk=0, k=None, v=None)
    assert lib.sp_attn_fwd(ctypes.byref(p), None, FAKE, None) == INVALID
    assert lib.sp_attn_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, None, None, None, FAKE, 1 << 40,
                           None) == INVALID


def test_attn_output_pointer_validation(lib):
    p = _params()
    assert lib.sp_attn_fwd(ctypes.byref(p), None, FAKE, None) == INVALID
    assert lib.sp_attn_fwd(ctypes.byref(p), FAKE, None, None) == INVALID
    assert lib.sp_attn_fwd(ctypes.byref(p), FAKE_ODD, FAKE, None) == MISALIGNED
    assert lib.sp_attn_fwd(None, FAKE, FAKE, None) == INVALID


def test_workspace_size_and_check(lib):
    p = _params(B=2, H=3, sq=200, d=64)
    rows = 256                                   # 200 rounded up to 128-row tiles
    up = lambda x: (x + 255) // 256 * 256
    expect = up(2 * 3 * rows * 64 * 4) + up(2 * 3 * 2 * rows * 4)
    assert lib.sp_attn_bwd_workspace_size(ctypes.byref(p)) == expect
    assert lib.sp_attn_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                           expect - 1, None) == WORKSPACE
    assert lib.sp_attn_bwd(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE + 16,
                           expect, None) == MISALIGNED


def test_empty_problems_launch_nothing(lib):
    # zero batch entries / heads / query rows: nothing to do, SP_OK without touching CUDA
    for kw in (dict(B=0), dict(H=0), dict(sq=0)):
        p = _params(**kw)
        assert lib.sp_attn_fwd(ctypes.byref(p), FAKE, FAKE, None) == OK


def _merge(**kw):
    p = binding.SpMergeParams()
    p.B, p.H, p.sq, p.d, p.init = 2, 3, 100, 128, 0
    p.o_part = p.o_acc = FAKE
    p.part_stride = (ctypes.c_int64 * 3)(100 * 3 * 128, 3 * 128, 128)
    p.lse_part = p.lse_acc = FAKE
    p.o_out = None
    p.out_stride = (ctypes.c_int64 * 3)(0, 0, 0)
    for k, v in kw.items():
        setattr(p, k, v)
    return p


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), UNSUPPORTED),
    (dict(sq=-1), INVALID),
    (dict(o_part=None), INVALID),
    (dict(lse_acc=None), INVALID),
    (dict(o_acc=FAKE_ODD), MISALIGNED),
    (dict(lse_part=FAKE + 2), MISALIGNED),
    (dict(part_stride=(ctypes.c_int64 * 3)(4, 4, 4)), MISALIGNED),
    (dict(o_out=FAKE_ODD), MISALIGNED),
    (dict(B=0), OK),                                  # nothing to merge, nothing launched
    (dict(sq=0, o_part=None, lse_part=None, o_acc=None, lse_acc=None), OK),   # empty: NULL ok
])
def test_merge_validation(lib, kw, code):
    p = _merge(**kw)
    assert lib.sp_attn_merge(ctypes.byref(p), None) == code


def test_merge_null_params(lib):
    assert lib.sp_attn_merge(None, None) == INVALID


def test_noalloc_refuses_dq_accumulation(lib):
    """The shared scratch carries no accumulation between calls."""
    p = _params(dq_accumulate=1)
    assert lib.sp_attn_bwd_noalloc(ctypes.byref(p), FAKE, FAKE, FAKE, FAKE, FAKE, FAKE,
                                   None) == INVALID


def test_packed_relayout_validation(lib):
    pout, keep = _arr(FAKE, FAKE * 2, FAKE * 3)
    f = lib.sp_relayout_seq2head_packed
    assert f(None, pout, 2, 1, 8, 4, 64, None) == INVALID           # no qkv buffer
    assert f(FAKE, pout, 2, 1, 8, 3, 64, None) == INVALID           # h % N
    assert f(FAKE_ODD, pout, 2, 1, 8, 4, 64, None) == MISALIGNED
    assert f(FAKE, pout, 2, 1, 8, 4, 3, None) == MISALIGNED         # parts 24 bytes apart
    pin, keep2 = _arr(FAKE, FAKE * 2, FAKE * 3)
    g = lib.sp_relayout_head2seq_packed
    assert g(pin, None, 2, 1, 8, 4, 64, None) == INVALID
    assert g(pin, FAKE_ODD, 2, 1, 8, 4, 64, None) == MISALIGNED


def test_linear_validation(lib):
    f, g = lib.sp_linear_fwd, lib.sp_linear_bwd
    assert f(FAKE, FAKE, FAKE, -1, 64, 64, None) == INVALID
    assert f(FAKE, FAKE, FAKE, 4, 0, 64, None) == INVALID
    assert f(FAKE, FAKE, FAKE, 4, 60, 64, None) == MISALIGNED          # rows not 16-byte
    assert f(None, FAKE, FAKE, 4, 64, 64, None) == INVALID
    assert f(FAKE_ODD, FAKE, FAKE, 4, 64, 64, None) == MISALIGNED
    assert f(FAKE, FAKE, FAKE, 0, 64, 64, None) == OK                  # no rows: nothing
    assert f(None, FAKE, None, 0, 64, 64, None) == OK                  # ... x, y may be NULL
    assert f(FAKE, None, FAKE, 0, 64, 64, None) == INVALID             # W is still required
    # no rows, dW accumulated into: unchanged, nothing launched; dy, x, dx may be NULL
    assert g(None, None, FAKE, None, FAKE, 0, 64, 64, 1, None) == OK
    assert g(None, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 0, None) == INVALID   # rows need dy
    assert g(FAKE, FAKE, FAKE, None, None, 4, 64, 64, 0, None) == INVALID   # nothing to do
    assert g(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 64, 64, 2, None) == INVALID
    assert g(FAKE, FAKE, FAKE, FAKE_ODD, FAKE, 4, 64, 64, 0, None) == MISALIGNED


def _host_params(**kw):
    p = binding.SpUlyssesHostParams()
    p.N, p.b, p.s, p.h, p.d, p.causal = 2, 1, 256, 4, 64, 1
    p.q = p.k = p.v = p.dout = p.o = p.dq = p.dk = p.dv = FAKE
    for name, val in kw.items():
        setattr(p, name, val)
    return p


def test_host_step_workspace_size(lib):
    f = lib.sp_ulysses_host_workspace_size
    # three slots of eight group tensors [b][s][h/N][d] bf16 and the lse, plus the
    # backward workspace of one group problem (fp32 dQ accumulator + two row statistics)
    N, b, s, h, d = 2, 1, 256, 4, 64
    tensor = b * s * (h // N) * d * 2
    lse = b * (h // N) * s * 4
    bwd = b * (h // N) * s * d * 4 + 2 * b * (h // N) * s * 4
    assert f(N, b, s, h, d, 1) == 3 * (8 * tensor + lse) + bwd
    assert f(0, b, s, h, d, 1) == 0
    assert f(3, b, s, h, d, 1) == 0            # s % N
    assert f(N, b, s, 3, d, 1) == 0            # h % N
    assert f(N, b, s, h, 96, 1) == 0           # head_dim
    assert f(N, b, s, h, d, 2) == 0            # causal flag


@pytest.mark.parametrize("kw,code", [
    ({"N": 0}, INVALID), ({"b": 0}, INVALID), ({"s": 255}, INVALID), ({"h": 3}, INVALID),
    ({"causal": 2}, INVALID), ({"d": 96}, UNSUPPORTED), ({"q": None}, INVALID),
    ({"dv": None}, INVALID),
])
def test_host_step_validation(lib, kw, code):
    """Every refusal that needs no GPU: sizes, flags and NULL pointers come first."""
    big = lib.sp_ulysses_host_workspace_size(2, 1, 256, 4, 64, 1)
    p = _host_params(**kw)
    assert lib.sp_ulysses_step_host(ctypes.byref(p), FAKE, big, None, FAKE, FAKE + 16) == code


def test_host_step_streams_and_workspace(lib):
    big = lib.sp_ulysses_host_workspace_size(2, 1, 256, 4, 64, 1)
    p = _host_params()
    f = lib.sp_ulysses_step_host
    assert f(None, FAKE, big, None, FAKE, FAKE + 16) == INVALID
    assert f(ctypes.byref(p), None, big, None, FAKE, FAKE + 16) == INVALID     # no workspace
    assert f(ctypes.byref(p), FAKE, big, None, None, FAKE + 16) == INVALID     # no h2d stream
    assert f(ctypes.byref(p), FAKE, big, None, FAKE, FAKE) == INVALID          # same stream twice
    assert f(ctypes.byref(p), FAKE, big, FAKE, FAKE, FAKE + 16) == INVALID     # copies on compute
    assert f(ctypes.byref(p), FAKE + 16, big, None, FAKE, FAKE + 32) == MISALIGNED
    pk = _host_params(key_len=FAKE + 2)
    assert f(ctypes.byref(pk), FAKE, big, None, FAKE, FAKE + 16) == MISALIGNED  # key_len
    assert f(ctypes.byref(p), FAKE, big - 1, None, FAKE, FAKE + 16) == WORKSPACE


def test_general_relayout_validation(lib):
    f = lib.sp_relayout
    shape = (ctypes.c_int64 * 4)(1, 8, 4, 64)
    assert f(FAKE, FAKE * 2, 2, None, 2, 1, None) == INVALID           # no shape
    assert f(FAKE, FAKE * 2, 0, shape, 2, 1, None) == INVALID          # N < 1
    assert f(FAKE, FAKE * 2, 2, shape, 0, 3, None) == UNSUPPORTED      # other dims
    assert f(FAKE, FAKE * 2, 2, shape, 2, 2, None) == UNSUPPORTED
    assert f(FAKE, FAKE * 2, 3, shape, 2, 1, None) == INVALID          # h = 4 not split by 3
    assert f(FAKE, FAKE * 2, 3, shape, 1, 2, None) == INVALID          # s = 8 not split by 3
    bad = (ctypes.c_int64 * 4)(1, 0, 4, 64)
    assert f(FAKE, FAKE * 2, 2, bad, 2, 1, None) == INVALID            # an empty dimension
    assert f(None, FAKE * 2, 2, shape, 2, 1, None) == INVALID
    assert f(FAKE_ODD, FAKE * 2, 2, shape, 2, 1, None) == MISALIGNED
