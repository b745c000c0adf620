"""GB300-native exact tiled attention: the FlashAttention-2 forward pass on sm_103a.

A thin ctypes binding over the C ABI in ``include/fa2.h`` (library
``libfa2_gb300.so``, built in-tree by ``exact_tiled_attention_fa2_gb300.build``).
Every step of the forward pass runs in the CUDA kernels; this module only
marshals torch tensors (device memory, streams) into pointers and sizes.
There is no CPU fallback: if the library is missing, calls raise.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa2_gb300.so")

FA2_FP16 = 0
FA2_BF16 = 1
FA2_OK = 0
FA2_ERR_INVALID_ARG = 1
FA2_ERR_UNSUPPORTED = 2
FA2_ERR_MISALIGNED = 3
FA2_ERR_CUDA = 4
FA2_ERR_DEVICE_TIMEOUT = 5
FA2_ERR_SCRATCH_LIMIT = 6
FA2_ERR_DEVICE_SEQLENS = 7
FA2_DECODE_MAX_Q = 8
FA2_NOALLOC_SCRATCH_BYTES = 32 << 20

_lib = None


class Fa2FwdParams(ctypes.Structure):
    """Mirror of ``fa2_fwd_params`` in include/fa2.h (checked against the library's sizeof)."""

    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("batch", ctypes.c_int), ("heads", ctypes.c_int),
        ("seqlen_q", ctypes.c_int), ("seqlen_k", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("scale", ctypes.c_float),
        ("window_left", ctypes.c_int), ("window_right", ctypes.c_int), ("prefix_len", ctypes.c_int),
        ("q_strides", ctypes.c_int64 * 3), ("k_strides", ctypes.c_int64 * 3),
        ("v_strides", ctypes.c_int64 * 3), ("o_strides", ctypes.c_int64 * 3),
        ("lse_strides", ctypes.c_int64 * 2),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("total_q", ctypes.c_int), ("total_k", ctypes.c_int),
    ]


class Fa2BwdParams(ctypes.Structure):
    """Mirror of ``fa2_bwd_params`` in include/fa2.h."""

    _fields_ = [
        ("fwd", Fa2FwdParams),
        ("dout", ctypes.c_void_p), ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
    ]


class Fa2Error(RuntimeError):
    """A nonzero fa2_status returned through the C ABI."""

    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s failed: %s (status %d)" % (where, fa2_status_string(code), code))


def load_library():
    """Load libfa2_gb300.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libfa2_gb300.so is not built (run `python -m exact_tiled_attention_fa2_gb300.build` "
                           "or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(LIB_PATH)
    vp, ci, cf, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa2_fwd.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.fa2_fwd.restype = ci
    lib.fa2_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, sz, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.fa2_fwd_host.restype = ci
    lib.fa2_fwd_host_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.fa2_fwd_host_workspace_bytes.restype = sz
    lib.fa2_fwd_host_noalloc.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.fa2_fwd_host_noalloc.restype = ci
    lib.fa2_bwd.argtypes = [vp] * 9 + [vp, sz, ci, ci, ci, ci, cf, ci, ci, vp]
    lib.fa2_bwd.restype = ci
    lib.fa2_bwd_workspace_bytes.argtypes = [ci, ci, ci, ci]
    lib.fa2_bwd_workspace_bytes.restype = sz
    lib.fa2_selftest_wait_timeout.argtypes = [ci, vp]
    lib.fa2_selftest_wait_timeout.restype = ci
    lib.fa2_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint32)]
    lib.fa2_get_device_status.restype = ci
    lib.fa2_status_string.argtypes = [ci]
    lib.fa2_status_string.restype = ctypes.c_char_p
    lib.fa2_version.argtypes = []
    lib.fa2_version.restype = ci
    lib.fa2_fwd_params_size.argtypes = []
    lib.fa2_fwd_params_size.restype = sz
    lib.fa2_fwd_ex.argtypes = [ctypes.POINTER(Fa2FwdParams), vp]
    lib.fa2_fwd_ex.restype = ci
    lib.fa2_decode.argtypes = [ctypes.POINTER(Fa2FwdParams), vp, sz, vp]
    lib.fa2_decode.restype = ci
    lib.fa2_decode_workspace_bytes.argtypes = [ctypes.POINTER(Fa2FwdParams)]
    lib.fa2_decode_workspace_bytes.restype = sz
    lib.fa2_bwd_ex.argtypes = [ctypes.POINTER(Fa2BwdParams), vp]
    lib.fa2_bwd_ex.restype = ci
    lib.fa2_bwd_ex_workspace_bytes.argtypes = [ctypes.POINTER(Fa2FwdParams)]
    lib.fa2_bwd_ex_workspace_bytes.restype = sz
    if lib.fa2_fwd_params_size() != ctypes.sizeof(Fa2FwdParams):
        raise RuntimeError("fa2_fwd_params layout mismatch: library %d bytes, binding %d bytes"
                           % (lib.fa2_fwd_params_size(), ctypes.sizeof(Fa2FwdParams)))
    _lib = lib
    return lib


def fa2_status_string(code: int) -> str:
    return load_library().fa2_status_string(int(code)).decode()


def fa2_version() -> int:
    return int(load_library().fa2_version())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float16:
        return FA2_FP16
    if t.dtype == torch.bfloat16:
        return FA2_BF16
    raise TypeError("q, k, v must be float16 or bfloat16, got %s" % t.dtype)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(int(stream.cuda_stream))


def fa2_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, stream=None):
    """Exact attention forward on CUDA tensors [B, H, N, d] (fp16/bf16, contiguous).

    Returns (o, lse): o [B,H,N,d] of q's dtype, lse [B,H,N] float32 (natural
    log).  ``scale`` defaults to 1/sqrt(d).  Asynchronous on ``stream``
    (default: torch's current stream).
    """
    import torch
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, N, d] shape")
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("fa2_fwd takes CUDA tensors; use fa2_fwd_host for host buffers")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous [B, H, N, d]")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    B, H, N, d = q.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    rc = load_library().fa2_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                B, H, N, d, float(scale), int(bool(causal)), _dtype_code(q),
                                _stream_handle(stream, q.device))
    if rc:
        raise Fa2Error(rc, "fa2_fwd")
    return o, lse


def _same_layout(a, b) -> bool:
    """Same shape, and the same stride wherever a dimension has more than one
    element (a size-1 dimension's stride addresses nothing)."""
    return a.shape == b.shape and all(sa == sb for sa, sb, n in zip(a.stride(), b.stride(), a.shape) if n > 1)


def _general_params(q, k, v, o, lse, scale, window_left, window_right, prefix_len, cu_seqlens_q, cu_seqlens_k,
                    max_seqlen_q, max_seqlen_k):
    """Marshal tensors into an Fa2FwdParams (allocating o and lse when not given)."""
    import torch
    packed = cu_seqlens_q is not None or cu_seqlens_k is not None
    if packed and (cu_seqlens_q is None or cu_seqlens_k is None):
        raise ValueError("give both cu_seqlens_q and cu_seqlens_k, or neither")
    for t in (q, k, v):
        if not t.is_cuda or t.stride(-1) != 1:
            raise ValueError("q, k, v must be CUDA tensors with a contiguous last dimension")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    d = q.shape[-1]
    p = Fa2FwdParams()
    if packed:
        if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or k.shape[1:] != q.shape[1:]:
            raise ValueError("packed q must be [total_q, H, d] and k, v [total_k, H, d]")
        for c in (cu_seqlens_q, cu_seqlens_k):
            if not c.is_cuda or c.dtype != torch.int32 or c.dim() != 1 or not c.is_contiguous():
                raise ValueError("cu_seqlens must be contiguous int32 CUDA tensors [B + 1]")
        total_q, H, _ = q.shape
        total_k = k.shape[0]
        B = cu_seqlens_q.numel() - 1
        if cu_seqlens_k.numel() != B + 1:
            raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
        if o is None:
            o = torch.empty_like(q, memory_format=torch.contiguous_format)
        if lse is None:
            lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
        p.batch, p.heads = B, H
        p.seqlen_q = total_q if max_seqlen_q is None else int(max_seqlen_q)
        p.seqlen_k = total_k if max_seqlen_k is None else int(max_seqlen_k)
        p.total_q, p.total_k = total_q, total_k
        for name, t in (("q_strides", q), ("k_strides", k), ("v_strides", v), ("o_strides", o)):
            getattr(p, name)[:] = [0, t.stride(1), t.stride(0)]
        p.lse_strides[:] = [0, lse.stride(0)]
        p.cu_seqlens_q = cu_seqlens_q.data_ptr()
        p.cu_seqlens_k = cu_seqlens_k.data_ptr()
    else:
        if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != d:
            raise ValueError("q must be [B, H, N_q, d] and k, v [B, H, N_k, d]")
        B, H, n_q, _ = q.shape
        if o is None:
            o = torch.empty(q.shape, dtype=q.dtype, device=q.device)
        if lse is None:
            lse = torch.empty((B, H, n_q), dtype=torch.float32, device=q.device)
        if lse.stride(-1) != 1:
            raise ValueError("lse must have a contiguous last dimension")
        p.batch, p.heads, p.seqlen_q, p.seqlen_k = B, H, n_q, k.shape[2]
        for name, t in (("q_strides", q), ("k_strides", k), ("v_strides", v), ("o_strides", o)):
            getattr(p, name)[:] = [t.stride(0), t.stride(1), t.stride(2)]
        p.lse_strides[:] = [lse.stride(0), lse.stride(1)]
    if o.dtype != q.dtype or o.stride(-1) != 1 or lse.dtype != torch.float32:
        raise ValueError("o must share q's dtype with a contiguous last dimension; lse must be float32")
    p.q, p.k, p.v, p.o, p.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()
    p.head_dim, p.dtype = d, _dtype_code(q)
    p.scale = 1.0 / float(d) ** 0.5 if scale is None else float(scale)
    p.window_left, p.window_right, p.prefix_len = int(window_left), int(window_right), int(prefix_len)
    return p, o, lse


def fa2_fwd_ex(q, k, v, o=None, lse=None, scale=None, window_left=-1, window_right=-1, prefix_len=0,
               cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, stream=None):
    """General forward (fa2_fwd_ex): strided views, N_q != N_k, band / prefix masks, packed batches.

    Unpacked: q [B, H, N_q, d], k and v [B, H, N_k, d], any CUDA views whose
    last dimension is contiguous (e.g. ``x.transpose(1, 2)`` of a [B, N, H, d]
    tensor); o (default: new contiguous [B, H, N_q, d]) and lse (default: new
    [B, H, N_q] float32) may be views too.

    Packed (cu_seqlens_q and cu_seqlens_k, int32 CUDA [B + 1]): q [total_q, H, d],
    k and v [total_k, H, d]; o [total_q, H, d] and lse [H, total_q] by default;
    ``max_seqlen_q`` (default: total_q) bounds every sequence's query count.

    Query i of a sequence sees key j iff j < prefix_len or
    i + off - window_left <= j <= i + off + window_right, off = N_k - N_q
    (-1 = unbounded).  causal is window (-1, 0).  Returns (o, lse).
    """
    p, o, lse = _general_params(q, k, v, o, lse, scale, window_left, window_right, prefix_len, cu_seqlens_q,
                                cu_seqlens_k, max_seqlen_q, None)
    rc = load_library().fa2_fwd_ex(ctypes.byref(p), _stream_handle(stream, q.device))
    if rc:
        raise Fa2Error(rc, "fa2_fwd_ex")
    return o, lse


def fa2_decode_workspace_bytes(q, k, v, **kw) -> int:
    """Workspace fa2_decode needs for these tensors and options (same keywords as fa2_decode)."""
    p, _, _ = _general_params(q, k, v, kw.get("o"), kw.get("lse"), kw.get("scale"), kw.get("window_left", -1),
                              kw.get("window_right", -1), kw.get("prefix_len", 0), kw.get("cu_seqlens_q"),
                              kw.get("cu_seqlens_k"), kw.get("max_seqlen_q"), kw.get("max_seqlen_k"))
    return int(load_library().fa2_decode_workspace_bytes(ctypes.byref(p)))


def fa2_decode(q, k, v, o=None, lse=None, workspace=None, scale=None, window_left=-1, window_right=-1, prefix_len=0,
               cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None, stream=None):
    """Decoding-regime forward (fa2_decode): at most FA2_DECODE_MAX_Q query rows per sequence.

    Same tensors and options as fa2_fwd_ex; ``workspace`` (a CUDA uint8
    tensor, allocated here when not given) holds the per-split partial
    states; packed batches take ``max_seqlen_k`` (default: total_k), the
    longest sequence's key count.  Returns (o, lse).
    """
    import torch
    p, o, lse = _general_params(q, k, v, o, lse, scale, window_left, window_right, prefix_len, cu_seqlens_q,
                                cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    lib = load_library()
    need = int(lib.fa2_decode_workspace_bytes(ctypes.byref(p)))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    rc = lib.fa2_decode(ctypes.byref(p), workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                        _stream_handle(stream, q.device))
    if rc:
        raise Fa2Error(rc, "fa2_decode")
    return o, lse


def fa2_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa2_bwd_workspace_bytes(B, H, N, d))


def fa2_bwd(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, workspace=None, scale=None, causal=False,
            stream=None):
    """Gradients (dq, dk, dv) of fa2_fwd for the upstream gradient dout (CUDA tensors, d = 64, 128 or 256)."""
    import torch
    for t in (q, k, v, o, dout):
        if not (t.is_cuda and t.is_contiguous() and t.dtype == q.dtype and t.shape == q.shape):
            raise ValueError("q, k, v, o, dout must be contiguous CUDA tensors of one shape and dtype")
    B, H, N, d = q.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    if workspace is None:
        workspace = torch.empty(fa2_bwd_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=q.device)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    rc = load_library().fa2_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                 dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), B, H, N, d, float(scale),
                                 int(bool(causal)), _dtype_code(q), _stream_handle(stream, q.device))
    if rc:
        raise Fa2Error(rc, "fa2_bwd")
    return dq, dk, dv


def fa2_bwd_ex(q, k, v, o, lse, dout, dq=None, dk=None, dv=None, workspace=None, scale=None, window_left=-1,
               window_right=-1, prefix_len=0, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None,
               max_seqlen_k=None, stream=None):
    """Gradients (dq, dk, dv) of fa2_fwd_ex (same tensors and options; o, lse its outputs).

    dout has o's layout; dq, dk, dv default to new tensors shaped like q, k,
    v (contiguous) and may be views.  Packed batches take ``max_seqlen_k``
    (default: total_k), the longest sequence's key count.  head dim 64, 128 or 256.
    """
    import torch
    p = Fa2BwdParams()
    fp, _, _ = _general_params(q, k, v, o, lse, scale, window_left, window_right, prefix_len, cu_seqlens_q,
                               cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    p.fwd = fp
    if not _same_layout(dout, o) or dout.dtype != o.dtype:
        raise ValueError("dout must have o's shape, strides and dtype")
    like = lambda t: torch.empty_strided(t.shape, t.stride(), dtype=t.dtype, device=t.device)
    dq = like(q) if dq is None else dq
    dk = like(k) if dk is None else dk
    dv = like(v) if dv is None else dv
    for g, t, name in ((dq, q, "dq"), (dk, k, "dk"), (dv, v, "dv")):
        if g.shape != t.shape or g.stride() != t.stride() or g.dtype != t.dtype:
            raise ValueError("%s must have the shape, strides and dtype of its primal tensor" % name)
    lib = load_library()
    if workspace is None:
        workspace = torch.empty(max(int(lib.fa2_bwd_ex_workspace_bytes(ctypes.byref(fp))), 256), dtype=torch.uint8,
                                device=q.device)
    p.dout, p.dq, p.dk, p.dv = dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    p.workspace, p.workspace_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = lib.fa2_bwd_ex(ctypes.byref(p), _stream_handle(stream, q.device))
    if rc:
        raise Fa2Error(rc, "fa2_bwd_ex")
    return dq, dk, dv


def _check_host_tensors(q, k, v, o, lse, where):
    """Shapes and dtypes of the host-buffer entry points' tensors, checked before
    any pointer is passed on: the library copies B*H*N*d 16-bit elements out of
    q, k, v and into o, and B*H*N floats into lse, so a smaller or differently
    typed tensor would be read or written past its end.  Returns (B, H, N, d)."""
    import torch
    for t in (q, k, v, o, lse):
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("%s takes contiguous host tensors" % where)
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape or o.shape != q.shape:
        raise ValueError("%s: q, k, v and o must share one [B, H, N, d] shape" % where)
    if q.element_size() != 2 or any(t.dtype != q.dtype for t in (k, v, o)):
        raise ValueError("%s: q, k, v and o must share one 16-bit dtype" % where)
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("%s: lse must be float32 of shape [B, H, N]" % where)
    return B, H, N, d


def fa2_fwd_host_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load_library().fa2_fwd_host_workspace_bytes(B, H, N, d))


def fa2_fwd_host(q, k, v, o, lse, workspace, scale=None, causal=False, dtype=None, stream=None):
    """End-to-end forward on HOST buffers (torch CPU tensors, ideally pinned).

    Copies q, k, v into ``workspace`` (a CUDA uint8 tensor of at least
    fa2_fwd_host_workspace_bytes bytes), runs the kernel, copies o and lse back
    into the given host tensors and synchronises the stream.
    """
    import torch
    B, H, N, d = _check_host_tensors(q, k, v, o, lse, "fa2_fwd_host")
    code = _dtype_code(q) if dtype is None else int(dtype)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    if not workspace.is_cuda or workspace.dtype != torch.uint8:
        raise ValueError("fa2_fwd_host: workspace must be a CUDA uint8 tensor")
    rc = load_library().fa2_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                     workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                     B, H, N, d, float(scale), int(bool(causal)), code,
                                     _stream_handle(stream, workspace.device))
    if rc:
        raise Fa2Error(rc, "fa2_fwd_host")
    return o, lse


def fa2_fwd_host_noalloc(q, k, v, o, lse, scale=None, causal=False, dtype=None, stream=None):
    """fa2_fwd_host without a caller-provided workspace, for callers that cannot allocate device memory.

    The device copies live in the library's static device array of
    FA2_NOALLOC_SCRATCH_BYTES bytes (held by every GPU that loads the library),
    so this call allocates nothing on the device.  Problems whose
    fa2_fwd_host_workspace_bytes exceed that size raise Fa2Error with
    FA2_ERR_SCRATCH_LIMIT.  Calls share the array: calls that overlap on the GPU
    race.  The first call on a device looks up the array's address there.
    """
    import torch
    B, H, N, d = _check_host_tensors(q, k, v, o, lse, "fa2_fwd_host_noalloc")
    code = _dtype_code(q) if dtype is None else int(dtype)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    rc = load_library().fa2_fwd_host_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                             lse.data_ptr(), B, H, N, d, float(scale), int(bool(causal)), code,
                                             _stream_handle(stream, torch.cuda.current_device()))
    if rc:
        raise Fa2Error(rc, "fa2_fwd_host_noalloc")
    return o, lse


def fa2_selftest_wait_timeout(limit_us: int = 2000, stream=None) -> None:
    """Launch the bounded-wait self-test (a wait that must expire after limit_us)."""
    import torch
    rc = load_library().fa2_selftest_wait_timeout(int(limit_us), _stream_handle(stream, torch.cuda.current_device()))
    if rc:
        raise Fa2Error(rc, "fa2_selftest_wait_timeout")


def fa2_get_device_status(stream=None):
    """Synchronise ``stream``; return (status, raw detail bits) and clear the device status word."""
    import torch
    detail = ctypes.c_uint32(0)
    rc = load_library().fa2_get_device_status(_stream_handle(stream, torch.cuda.current_device()),
                                              ctypes.byref(detail))
    return rc, int(detail.value)
