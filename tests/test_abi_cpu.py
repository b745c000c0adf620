"""The C-ABI library loads without a GPU, exports every symbol include/*.h
declares, and rejects bad arguments before making any CUDA call.  CPU only:
no call here ever reaches a kernel launch (every call carries an invalid
argument), so the file is also safe on a GPU machine."""
import ctypes
import glob
import os
import re

import pytest

import exact_tiled_attention_fa2_gb300 as fa2
from exact_tiled_attention_fa2_gb300 import build as fa2_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fa2_build.build()
    return fa2.load_library()


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(fa2_\w+)\s*\(", text, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


def test_header_declares_entry_points():
    names = _declared_functions()
    for required in ("fa2_fwd", "fa2_fwd_host", "fa2_fwd_host_workspace_bytes", "fa2_get_device_status",
                     "fa2_status_string", "fa2_version", "fa2_selftest_wait_timeout", "fa2_bwd",
                     "fa2_bwd_workspace_bytes", "fa2_fwd_host_noalloc", "fa2_fwd_ex", "fa2_bwd_ex",
                     "fa2_decode"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_status_strings(lib):
    for code in range(8):
        s = fa2.fa2_status_string(code)
        assert isinstance(s, str) and s
    assert fa2.fa2_status_string(0) == "ok"
    assert "unknown" in fa2.fa2_status_string(99)
    assert fa2.fa2_version() >= 100


# Pointer values below are never dereferenced: each call fails argument checks first.
A = 0x10000  # 16-byte aligned stand-ins
GOOD = dict(B=1, H=2, N=64, d=64, scale=0.125, causal=0, dtype=0)


def _call(lib, q=A, k=2 * A, v=3 * A, o=4 * A, lse=5 * A, **kw):
    a = dict(GOOD)
    a.update(kw)
    return lib.fa2_fwd(q, k, v, o, lse, a["B"], a["H"], a["N"], a["d"], a["scale"], a["causal"], a["dtype"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), fa2.FA2_ERR_INVALID_ARG),
    (dict(dtype=-1), fa2.FA2_ERR_INVALID_ARG),
    (dict(B=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(H=-3), fa2.FA2_ERR_INVALID_ARG),
    (dict(N=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(causal=2), fa2.FA2_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa2.FA2_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa2.FA2_ERR_INVALID_ARG),
    (dict(scale=float("-inf")), fa2.FA2_ERR_INVALID_ARG),
    (dict(d=32), fa2.FA2_ERR_UNSUPPORTED),
    (dict(d=96), fa2.FA2_ERR_UNSUPPORTED),
    (dict(d=512), fa2.FA2_ERR_UNSUPPORTED),
    (dict(N=2 ** 30, H=2 ** 10), fa2.FA2_ERR_UNSUPPORTED),
])
def test_bad_sizes_rejected(lib, kw, code):
    assert _call(lib, **kw) == code


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_null_pointers_rejected(lib, which):
    assert _call(lib, **{which: 0}) == fa2.FA2_ERR_INVALID_ARG


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_misaligned_pointers_rejected(lib, which):
    base = {"q": A, "k": 2 * A, "v": 3 * A, "o": 4 * A, "lse": 5 * A}[which]
    assert _call(lib, **{which: base + 8}) == fa2.FA2_ERR_MISALIGNED


def test_overlapping_outputs_rejected(lib):
    # o overlapping k, lse overlapping q, o overlapping lse
    assert _call(lib, o=2 * A + 1024) == fa2.FA2_ERR_INVALID_ARG
    assert _call(lib, lse=A + 4096) == fa2.FA2_ERR_INVALID_ARG
    assert _call(lib, lse=4 * A + 16) == fa2.FA2_ERR_INVALID_ARG


def test_host_entry_point_checks(lib):
    ws = fa2.fa2_fwd_host_workspace_bytes(1, 2, 64, 64)
    assert ws == 4 * 16384 + 512
    assert fa2.fa2_fwd_host_workspace_bytes(0, 2, 64, 64) == 0
    f = lib.fa2_fwd_host
    # workspace too small, misaligned workspace, null host pointer, bad dtype
    assert f(A, A, A, A, A, 6 * A, ws - 1, 1, 2, 64, 64, 0.125, 0, 0, None) == fa2.FA2_ERR_INVALID_ARG
    assert f(A, A, A, A, A, 6 * A + 16, ws, 1, 2, 64, 64, 0.125, 0, 0, None) == fa2.FA2_ERR_MISALIGNED
    assert f(0, A, A, A, A, 6 * A, ws, 1, 2, 64, 64, 0.125, 0, 0, None) == fa2.FA2_ERR_INVALID_ARG
    assert f(A, A, A, A, A, 6 * A, ws, 1, 2, 64, 64, 0.125, 0, 5, None) == fa2.FA2_ERR_INVALID_ARG


def test_noalloc_host_entry_point_checks(lib):
    # every check runs before any CUDA call, so the stand-in pointers are never touched
    f = lib.fa2_fwd_host_noalloc
    assert f(A, A, A, A, 0, 1, 2, 64, 64, 0.125, 0, 0, None) == fa2.FA2_ERR_INVALID_ARG     # null lse
    assert f(0, A, A, A, A, 1, 2, 64, 64, 0.125, 0, 0, None) == fa2.FA2_ERR_INVALID_ARG     # null q
    assert f(A, A, A, A, A, 1, 2, 64, 96, 0.125, 0, 0, None) == fa2.FA2_ERR_UNSUPPORTED     # head dim 96
    assert f(A, A, A, A, A, 1, 2, 64, 64, float("nan"), 0, 0, None) == fa2.FA2_ERR_INVALID_ARG
    # B1 H16 N4096 d128 needs 64 MiB + 256 KiB of staging, beyond the 32 MiB array
    assert fa2.fa2_fwd_host_workspace_bytes(1, 16, 4096, 128) > fa2.FA2_NOALLOC_SCRATCH_BYTES
    assert f(A, A, A, A, A, 1, 16, 4096, 128, 0.088, 1, 0, None) == fa2.FA2_ERR_SCRATCH_LIMIT


def test_host_wrappers_check_shapes_and_dtypes():
    # the Python host wrappers refuse tensors the library would read or write past their ends
    import torch
    q = torch.zeros((1, 2, 64, 64), dtype=torch.float16)
    lse = torch.zeros((1, 2, 64), dtype=torch.float32)
    small = torch.zeros((1, 2, 32, 64), dtype=torch.float16)
    bad = [
        dict(k=small),                                          # k smaller than q
        dict(o=small),                                          # o smaller than q
        dict(o=torch.zeros((1, 2, 64, 64), dtype=torch.float32)),   # fp32 o
        dict(v=q.to(torch.bfloat16)),                           # mixed dtypes
        dict(lse=torch.zeros((1, 2, 64), dtype=torch.float16)),     # 16-bit lse
        dict(lse=torch.zeros((1, 2, 63), dtype=torch.float32)),     # short lse
        dict(q=torch.zeros((2, 64, 64), dtype=torch.float16)),      # not 4-D
    ]
    for kw in bad:
        t = dict(q=q, k=q.clone(), v=q.clone(), o=q.clone(), lse=lse)
        t.update(kw)
        with pytest.raises(ValueError):
            fa2.fa2_fwd_host_noalloc(t["q"], t["k"], t["v"], t["o"], t["lse"])
        with pytest.raises(ValueError):
            fa2.fa2_fwd_host(t["q"], t["k"], t["v"], t["o"], t["lse"], torch.zeros(16, dtype=torch.uint8))


def test_selftest_limit_checked(lib):
    assert lib.fa2_selftest_wait_timeout(0, None) == fa2.FA2_ERR_INVALID_ARG
    assert lib.fa2_selftest_wait_timeout(1000001, None) == fa2.FA2_ERR_INVALID_ARG


# ---------------------------------------------------------------- fa2_fwd_ex argument checks


def _params(**kw):
    """A valid contiguous [1, 2, 64, 64] problem (pointers are stand-ins), then overrides."""
    p = fa2.Fa2FwdParams()
    p.q, p.k, p.v, p.o, p.lse = A, 2 * A, 3 * A, 4 * A, 5 * A
    p.batch, p.heads, p.seqlen_q, p.seqlen_k, p.head_dim = 1, 2, 64, 64, 64
    p.dtype, p.scale = 0, 0.125
    p.window_left, p.window_right, p.prefix_len = -1, -1, 0
    for name in ("q_strides", "k_strides", "v_strides", "o_strides"):
        getattr(p, name)[:] = [2 * 64 * 64, 64 * 64, 64]
    p.lse_strides[:] = [128, 64]
    for key, val in kw.items():
        if isinstance(val, list):
            getattr(p, key)[:] = val
        else:
            setattr(p, key, val)
    return p


def _ex(lib, **kw):
    return lib.fa2_fwd_ex(ctypes.byref(_params(**kw)), None)


def test_params_struct_matches_library(lib):
    assert lib.fa2_fwd_params_size() == ctypes.sizeof(fa2.Fa2FwdParams)


def test_ex_null_params(lib):
    assert lib.fa2_fwd_ex(None, None) == fa2.FA2_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,code", [
    (dict(window_left=-2), fa2.FA2_ERR_INVALID_ARG),
    (dict(window_right=-5), fa2.FA2_ERR_INVALID_ARG),
    (dict(prefix_len=-1), fa2.FA2_ERR_INVALID_ARG),
    (dict(seqlen_k=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(seqlen_q=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(head_dim=96), fa2.FA2_ERR_UNSUPPORTED),
    (dict(dtype=3), fa2.FA2_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa2.FA2_ERR_INVALID_ARG),
    (dict(q_strides=[8192, 4096, 68]), fa2.FA2_ERR_MISALIGNED),      # row stride not a multiple of 8
    (dict(k_strides=[8192, 4100, 64]), fa2.FA2_ERR_MISALIGNED),      # head stride not a multiple of 8
    (dict(v_strides=[8192, 0, 64]), fa2.FA2_ERR_INVALID_ARG),        # zero stride on a dimension of size 2
    (dict(o_strides=[8192, 4096, -64]), fa2.FA2_ERR_INVALID_ARG),    # negative stride
    (dict(q_strides=[8192, 4096, 1 << 40]), fa2.FA2_ERR_INVALID_ARG),
    (dict(lse=5 * A + 2), fa2.FA2_ERR_MISALIGNED),
    (dict(o=4 * A + 8), fa2.FA2_ERR_MISALIGNED),
    (dict(o=2 * A + 2048), fa2.FA2_ERR_INVALID_ARG),                 # o inside k
    (dict(lse=3 * A + 4096), fa2.FA2_ERR_INVALID_ARG),               # lse inside v
    (dict(lse=4 * A + 8192), fa2.FA2_ERR_INVALID_ARG),               # lse inside o
    (dict(cu_seqlens_q=7 * A), fa2.FA2_ERR_INVALID_ARG),             # only one offsets array
    (dict(cu_seqlens_q=7 * A, cu_seqlens_k=8 * A, total_q=0, total_k=64), fa2.FA2_ERR_INVALID_ARG),
    (dict(cu_seqlens_q=7 * A + 2, cu_seqlens_k=8 * A, total_q=64, total_k=64), fa2.FA2_ERR_MISALIGNED),
    (dict(q=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(batch=2 ** 20, heads=2 ** 10, seqlen_q=2 ** 20), fa2.FA2_ERR_UNSUPPORTED),
])
def test_ex_bad_arguments_rejected(lib, kw, code):
    assert _ex(lib, **kw) == code


def test_ex_stride_of_size_one_dimension_is_ignored(lib):
    # batch = 1: an unaligned batch stride is never used, so the call gets past the
    # stride checks and fails on the (deliberate) overlap of o with k instead
    assert _ex(lib, q_strides=[3, 4096, 64], o=2 * A + 2048) == fa2.FA2_ERR_INVALID_ARG
    assert _ex(lib, q_strides=[3, 4096, 64], batch=2, o=2 * A + 2048) == fa2.FA2_ERR_MISALIGNED


def test_ex_bnhd_output_overlap_detected(lib):
    # o as a [B, N, H, d] layout (row stride H*d, head stride d) reaching into lse
    assert _ex(lib, o_strides=[8192, 64, 128], lse=4 * A + 16000) == fa2.FA2_ERR_INVALID_ARG


# ---------------------------------------------------------------- fa2_decode argument checks


def _decode(lib, ws=9 * A, ws_bytes=1 << 20, **kw):
    kw = dict(dict(seqlen_q=1), **kw)
    return lib.fa2_decode(ctypes.byref(_params(**kw)), ws, ws_bytes, None)


def test_decode_workspace_plan_is_device_independent(lib):
    # B1 H32 N_k 16384 d128: 304 // 32 = 9 splits of ceil(16384 / 9) = 1821 -> 1856 keys (a multiple
    # of the 64-key stage); 288 slots x (128 + 2) floats, each array 256-byte aligned
    p = _params(batch=1, heads=32, seqlen_q=1, seqlen_k=16384, head_dim=128)
    assert lib.fa2_decode_workspace_bytes(ctypes.byref(p)) == 288 * 128 * 4 + 2304
    # more heads than two per SM: one split each; short caches: no split below 256 keys
    p = _params(batch=4, heads=128, seqlen_q=2, seqlen_k=1000, head_dim=64)
    assert lib.fa2_decode_workspace_bytes(ctypes.byref(p)) == 512 * 2 * 64 * 4 + 512 * 2 * 8
    p = _params(batch=1, heads=2, seqlen_q=1, seqlen_k=600, head_dim=256)
    slots = 2 * 3   # ceil(600 / 256) = 3 splits of 224 keys
    assert lib.fa2_decode_workspace_bytes(ctypes.byref(p)) == (slots * 256 * 4 + 255) // 256 * 256 + 256
    assert lib.fa2_decode_workspace_bytes(ctypes.byref(_params(seqlen_q=9))) == 0
    assert lib.fa2_decode_workspace_bytes(None) == 0


def test_decode_plan_skips_keys_no_row_sees(lib):
    # window (4095, 0), one row vs 16384 keys: keys below 16384 - 1 - 4095 = 12288 are seen by no row,
    # so 9 splits cover 4096 keys: ceil(4096 / 9) = 456 -> 512 (a multiple of 64), i.e. 8 chunks
    p = _params(batch=1, heads=32, seqlen_q=1, seqlen_k=16384, head_dim=128, window_left=4095, window_right=0)
    assert lib.fa2_decode_workspace_bytes(ctypes.byref(p)) == 32 * 8 * 128 * 4 + 32 * 8 * 2 * 4
    # a prefix keeps every chunk from key 0 (the plan of the unwindowed call)
    p = _params(batch=1, heads=32, seqlen_q=1, seqlen_k=16384, head_dim=128, window_left=4095, window_right=0,
                prefix_len=16)
    assert lib.fa2_decode_workspace_bytes(ctypes.byref(p)) == 288 * 128 * 4 + 2304


@pytest.mark.parametrize("kw,code", [
    (dict(seqlen_q=9), fa2.FA2_ERR_UNSUPPORTED),
    (dict(seqlen_q=0), fa2.FA2_ERR_UNSUPPORTED),
    (dict(head_dim=96), fa2.FA2_ERR_UNSUPPORTED),
    (dict(ws=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(ws=9 * A + 128), fa2.FA2_ERR_MISALIGNED),
    (dict(ws_bytes=100), fa2.FA2_ERR_INVALID_ARG),
    (dict(window_left=-3), fa2.FA2_ERR_INVALID_ARG),
    (dict(k_strides=[8192, 4096, 60]), fa2.FA2_ERR_MISALIGNED),
    (dict(ws=4 * A), fa2.FA2_ERR_INVALID_ARG),                      # workspace over o
    (dict(ws=A), fa2.FA2_ERR_INVALID_ARG),                          # workspace over q
])
def test_decode_bad_arguments_rejected(lib, kw, code):
    assert _decode(lib, **kw) == code


def test_decode_null_params(lib):
    assert lib.fa2_decode(None, 9 * A, 1 << 20, None) == fa2.FA2_ERR_INVALID_ARG


# ---------------------------------------------------------------- fa2_bwd_ex argument checks


def _bwd(lib, dout=6 * A, dq=7 * A, dk=8 * A, dv=9 * A, ws=10 * A, ws_bytes=1 << 20, **kw):
    b = fa2.Fa2BwdParams()
    b.fwd = _params(**kw)
    b.dout, b.dq, b.dk, b.dv, b.workspace, b.workspace_bytes = dout, dq, dk, dv, ws, ws_bytes
    return lib.fa2_bwd_ex(ctypes.byref(b), None)


def test_bwd_ex_workspace_plan(lib):
    # [1, 2, 64, 64]: fp32 accumulator 2 x 64 x 64 x 4 bytes + D 2 x 64 x 4 bytes (256-byte aligned)
    assert lib.fa2_bwd_ex_workspace_bytes(ctypes.byref(_params())) == 32768 + 512
    # d = 256: the same layout with 256 columns
    assert lib.fa2_bwd_ex_workspace_bytes(ctypes.byref(_params(head_dim=256))) == 131072 + 512
    assert lib.fa2_bwd_ex_workspace_bytes(ctypes.byref(_params(head_dim=96))) == 0
    assert lib.fa2_bwd_ex_workspace_bytes(None) == 0
    # the contiguous entry point asks for the same amount
    assert fa2.fa2_bwd_workspace_bytes(1, 2, 64, 64) == 32768 + 512


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), fa2.FA2_ERR_UNSUPPORTED),
    (dict(dq=0), fa2.FA2_ERR_INVALID_ARG),
    (dict(dout=6 * A + 8), fa2.FA2_ERR_MISALIGNED),
    (dict(ws=10 * A + 64), fa2.FA2_ERR_MISALIGNED),
    (dict(ws_bytes=1000), fa2.FA2_ERR_INVALID_ARG),
    (dict(dq=A + 512), fa2.FA2_ERR_INVALID_ARG),           # dq over q
    (dict(dk=6 * A), fa2.FA2_ERR_INVALID_ARG),             # dk over dout
    (dict(dv=7 * A + 1024), fa2.FA2_ERR_INVALID_ARG),      # dv over dq
    (dict(ws=8 * A), fa2.FA2_ERR_INVALID_ARG),             # workspace over dk
    (dict(window_left=-7), fa2.FA2_ERR_INVALID_ARG),
])
def test_bwd_ex_bad_arguments_rejected(lib, kw, code):
    assert _bwd(lib, **kw) == code


def test_bwd_ex_null_params(lib):
    assert lib.fa2_bwd_ex(None, None) == fa2.FA2_ERR_INVALID_ARG


def test_same_layout_ignores_strides_of_size_one_dimensions():
    """dout must share o's layout; a size-1 dimension's stride addresses
    nothing, so it may differ (numpy gives a transposed [T, 1, d] view the
    stride of the dimension it came from)."""
    import torch
    from exact_tiled_attention_fa2_gb300 import _same_layout
    a = torch.empty(5, 1, 8)
    b = torch.empty(5 * 40).as_strided((5, 1, 8), (8, 40, 1))
    assert a.stride() != b.stride() and _same_layout(a, b)
    c = torch.empty(5 * 16).as_strided((5, 1, 8), (16, 8, 1))   # rows 16 apart, not 8
    assert not _same_layout(a, c)
    assert not _same_layout(a, torch.empty(5, 2, 8))
