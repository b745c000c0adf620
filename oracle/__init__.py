"""CPU oracle for exact softmax attention -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports it and shares no code with it.

``attention_rows`` / ``attention_fwd`` call the plain fp64 C implementation in
``attention_oracle.c`` (the definition S = scale*QK^T, P = softmax_row(S),
O = PV, L = m + ln sum exp(S - m), from the Flash Attention 2 page "Standard
Attention" and FlashAttention V2 in depth section 6.1).  ``tiled_reference``
restates the tiled online-softmax algorithm of FlashAttention V2 in depth
section 6.1 in numpy; tests use it to check that tiling is exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

FP16 = 0
BF16 = 1


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` (gcc, OpenMP)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        p16 = ctypes.POINTER(ctypes.c_uint16)
        pd = ctypes.POINTER(ctypes.c_double)
        pi64 = ctypes.POINTER(ctypes.c_int64)
        i64 = ctypes.c_int64
        lib.oracle_attention_rows.argtypes = [p16, p16, p16, ctypes.c_int, i64, i64, i64, i64,
                                              ctypes.c_double, ctypes.c_int, pi64, pi64, i64, pd, pd,
                                              ctypes.c_int]
        lib.oracle_attention_rows.restype = ctypes.c_int
        lib.oracle_attention_fwd.argtypes = [p16, p16, p16, ctypes.c_int, i64, i64, i64, i64,
                                             ctypes.c_double, ctypes.c_int, pd, pd, ctypes.c_int]
        lib.oracle_attention_fwd.restype = ctypes.c_int
        lib.oracle_widen.argtypes = [p16, ctypes.c_int, i64, pd]
        lib.oracle_widen.restype = ctypes.c_int
        lib.oracle_attention_fwd_f64.argtypes = [pd, pd, pd, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int, pd, pd]
        lib.oracle_attention_fwd_f64.restype = ctypes.c_int
        lib.oracle_attention_bwd_f64.argtypes = [pd, pd, pd, pd, i64, i64, i64, i64, ctypes.c_double, ctypes.c_int,
                                                 pd, pd, pd, pd, ctypes.c_int]
        lib.oracle_attention_bwd_f64.restype = ctypes.c_int
        lib.oracle_attention_bwd.argtypes = [p16, p16, p16, p16, ctypes.c_int, i64, i64, i64, i64, ctypes.c_double,
                                             ctypes.c_int, pd, pd, pd, pd, ctypes.c_int]
        lib.oracle_attention_bwd.restype = ctypes.c_int
        lib.oracle_attention_bwd_rows.argtypes = [p16, p16, p16, p16, ctypes.c_int, i64, i64, i64, i64,
                                                  ctypes.c_double, ctypes.c_int, pi64, pi64, i64, pd, pd,
                                                  ctypes.c_int]
        lib.oracle_attention_bwd_rows.restype = ctypes.c_int
        lib.oracle_attention_bwd_keys.argtypes = [p16, p16, p16, p16, ctypes.c_int, i64, i64, i64, i64,
                                                  ctypes.c_double, ctypes.c_int, i64, pi64, i64, pd, pd,
                                                  ctypes.c_int]
        lib.oracle_attention_bwd_keys.restype = ctypes.c_int
        lib.oracle_attention_fwd_masked.argtypes = [p16, p16, p16, ctypes.c_int, i64, i64, i64, i64, i64,
                                                    ctypes.c_double, i64, i64, i64, pd, pd, ctypes.c_int]
        lib.oracle_attention_fwd_masked.restype = ctypes.c_int
        lib.oracle_attention_rows_masked.argtypes = [p16, p16, p16, ctypes.c_int, i64, i64, i64, i64, i64,
                                                     ctypes.c_double, i64, i64, i64, pi64, pi64, i64, pd, pd,
                                                     ctypes.c_int]
        lib.oracle_attention_rows_masked.restype = ctypes.c_int
        lib.oracle_attention_fwd_masked_f64.argtypes = [pd, pd, pd, i64, i64, i64, i64, i64, ctypes.c_double, i64, i64,
                                                        i64, pd, pd]
        lib.oracle_attention_fwd_masked_f64.restype = ctypes.c_int
        lib.oracle_attention_bwd_masked_f64.argtypes = [pd, pd, pd, pd, i64, i64, i64, i64, i64, ctypes.c_double, i64,
                                                        i64, i64, pd, pd, pd, pd, ctypes.c_int]
        lib.oracle_attention_bwd_masked_f64.restype = ctypes.c_int
        lib.oracle_attention_bwd_masked.argtypes = [p16, p16, p16, p16, ctypes.c_int, i64, i64, i64, i64, i64,
                                                    ctypes.c_double, i64, i64, i64, pd, pd, pd, pd, ctypes.c_int]
        lib.oracle_attention_bwd_masked.restype = ctypes.c_int
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are 16-bit bit patterns (uint16), got %s" % a.dtype)
    return a


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def max_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_load().oracle_max_threads())


def widen(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact fp16/bf16 -> float64 widening done by the oracle's own decoder."""
    bits = _bits(bits)
    out = np.empty(bits.shape, dtype=np.float64)
    rc = _load().oracle_widen(_ptr(bits, ctypes.c_uint16), int(dtype), bits.size, _ptr(out, ctypes.c_double))
    if rc:
        raise ValueError("oracle_widen failed (%d)" % rc)
    return out


def attention_fwd(q, k, v, dtype: int, scale: float, causal: bool, threads: int = 0):
    """Full O [B,H,N,d] and L [B,H,N] in float64 from 16-bit bit patterns [B,H,N,d]."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B,H,N,d] shape")
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d), dtype=np.float64)
    lse = np.empty((B, H, N), dtype=np.float64)
    rc = _load().oracle_attention_fwd(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                      _ptr(v, ctypes.c_uint16), int(dtype), B, H, N, d, float(scale),
                                      int(bool(causal)), _ptr(o, ctypes.c_double),
                                      _ptr(lse, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_fwd failed (%d)" % rc)
    return o, lse


def attention_rows(q, k, v, dtype: int, scale: float, causal: bool, bh_idx, row_idx, threads: int = 0):
    """O rows [count, d] and L [count] for the (bh, row) samples, float64."""
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, N, d = q.shape
    bh_idx = np.ascontiguousarray(bh_idx, dtype=np.int64)
    row_idx = np.ascontiguousarray(row_idx, dtype=np.int64)
    count = bh_idx.size
    o = np.empty((count, d), dtype=np.float64)
    lse = np.empty((count,), dtype=np.float64)
    rc = _load().oracle_attention_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                       _ptr(v, ctypes.c_uint16), int(dtype), B, H, N, d, float(scale),
                                       int(bool(causal)), _ptr(bh_idx, ctypes.c_int64),
                                       _ptr(row_idx, ctypes.c_int64), count, _ptr(o, ctypes.c_double),
                                       _ptr(lse, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_rows failed (%d)" % rc)
    return o, lse


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def attention_fwd_f64(q, k, v, scale: float, causal: bool):
    """Forward on float64 inputs [B,H,N,d]: (O, L) by the same definition."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, d = q.shape
    o = np.empty((B, H, N, d))
    lse = np.empty((B, H, N))
    rc = _load().oracle_attention_fwd_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                          _ptr(v, ctypes.c_double), B, H, N, d, float(scale), int(bool(causal)),
                                          _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc:
        raise ValueError("oracle_attention_fwd_f64 failed (%d)" % rc)
    return o, lse


def attention_bwd_f64(q, k, v, dout, scale: float, causal: bool, threads: int = 0):
    """Gradients (dQ, dK, dV, D) of the forward pass for upstream dO, float64 inputs [B,H,N,d]."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, N, d = q.shape
    dq, dk, dv = (np.empty((B, H, N, d)) for _ in range(3))
    delta = np.empty((B, H, N))
    rc = _load().oracle_attention_bwd_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                          _ptr(v, ctypes.c_double), _ptr(dout, ctypes.c_double), B, H, N, d,
                                          float(scale), int(bool(causal)), _ptr(dq, ctypes.c_double),
                                          _ptr(dk, ctypes.c_double), _ptr(dv, ctypes.c_double),
                                          _ptr(delta, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_bwd_f64 failed (%d)" % rc)
    return dq, dk, dv, delta


def attention_bwd(q, k, v, dout, dtype: int, scale: float, causal: bool, threads: int = 0):
    """Gradients (dQ, dK, dV, D) from 16-bit bit patterns [B,H,N,d], float64 results."""
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, N, d = q.shape
    dq, dk, dv = (np.empty((B, H, N, d)) for _ in range(3))
    delta = np.empty((B, H, N))
    rc = _load().oracle_attention_bwd(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                                      _ptr(dout, ctypes.c_uint16), int(dtype), B, H, N, d, float(scale),
                                      int(bool(causal)), _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                      _ptr(dv, ctypes.c_double), _ptr(delta, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_bwd failed (%d)" % rc)
    return dq, dk, dv, delta


def attention_bwd_rows(q, k, v, dout, dtype: int, scale: float, causal: bool, bh_idx, row_idx, threads: int = 0):
    """dQ rows [count, d] and D [count] of the backward at the sampled (bh, row)
    pairs, from 16-bit bit patterns [B,H,N,d], float64: the rows pass of
    attention_bwd for those rows only."""
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, N, d = q.shape
    bh_idx = np.ascontiguousarray(bh_idx, dtype=np.int64)
    row_idx = np.ascontiguousarray(row_idx, dtype=np.int64)
    count = bh_idx.size
    if row_idx.size != count:
        raise ValueError("bh_idx and row_idx must have one length")
    dq = np.empty((count, d))
    delta = np.empty((count,))
    rc = _load().oracle_attention_bwd_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                           _ptr(v, ctypes.c_uint16), _ptr(dout, ctypes.c_uint16), int(dtype), B, H,
                                           N, d, float(scale), int(bool(causal)), _ptr(bh_idx, ctypes.c_int64),
                                           _ptr(row_idx, ctypes.c_int64), count, _ptr(dq, ctypes.c_double),
                                           _ptr(delta, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_bwd_rows failed (%d)" % rc)
    return dq, delta


def attention_bwd_keys(q, k, v, dout, dtype: int, scale: float, causal: bool, bh: int, key_idx, threads: int = 0):
    """dK and dV rows [count, d] of the backward at the sampled keys of slice
    bh (= b * H + h), from 16-bit bit patterns [B,H,N,d], float64: the keys
    pass of attention_bwd for those keys, over every row that sees them."""
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, N, d = q.shape
    key_idx = np.ascontiguousarray(key_idx, dtype=np.int64)
    count = key_idx.size
    dk = np.empty((count, d))
    dv = np.empty((count, d))
    rc = _load().oracle_attention_bwd_keys(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                           _ptr(v, ctypes.c_uint16), _ptr(dout, ctypes.c_uint16), int(dtype), B, H,
                                           N, d, float(scale), int(bool(causal)), int(bh),
                                           _ptr(key_idx, ctypes.c_int64), count, _ptr(dk, ctypes.c_double),
                                           _ptr(dv, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_bwd_keys failed (%d)" % rc)
    return dk, dv


def _masked_shapes(q, k, v):
    q, k, v = _bits(q), _bits(k), _bits(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k, v must be [B,H,Nk,d] with q's B, H, d")
    return q, k, v, B, H, Nq, Nk, d


def attention_fwd_masked(q, k, v, dtype: int, scale: float, window_left: int = -1, window_right: int = -1,
                         prefix_len: int = 0, threads: int = 0):
    """Forward with a band / prefix mask and N_q != N_k: q [B,H,Nq,d], k, v [B,H,Nk,d] (16-bit bit patterns).

    Key j is visible to query i iff j < prefix_len, or j >= i + (Nk - Nq) -
    window_left and j <= i + (Nk - Nq) + window_right (a negative window is
    unbounded on that side; causal is window_right = 0).  Rows with nothing
    visible: O = 0, L = -inf.  Returns float64 (O [B,H,Nq,d], L [B,H,Nq]).
    """
    q, k, v, B, H, Nq, Nk, d = _masked_shapes(q, k, v)
    o = np.empty((B, H, Nq, d))
    lse = np.empty((B, H, Nq))
    rc = _load().oracle_attention_fwd_masked(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                             _ptr(v, ctypes.c_uint16), int(dtype), B, H, Nq, Nk, d, float(scale),
                                             int(window_left), int(window_right), int(prefix_len),
                                             _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_fwd_masked failed (%d)" % rc)
    return o, lse


def attention_rows_masked(q, k, v, dtype: int, scale: float, bh_idx, row_idx, window_left: int = -1,
                          window_right: int = -1, prefix_len: int = 0, threads: int = 0):
    """attention_fwd_masked at sampled (bh, row) pairs: O rows [count, d] and L [count], float64."""
    q, k, v, B, H, Nq, Nk, d = _masked_shapes(q, k, v)
    bh_idx = np.ascontiguousarray(bh_idx, dtype=np.int64)
    row_idx = np.ascontiguousarray(row_idx, dtype=np.int64)
    count = bh_idx.size
    if row_idx.size != count:
        raise ValueError("bh_idx and row_idx must have one length")
    o = np.empty((count, d))
    lse = np.empty((count,))
    rc = _load().oracle_attention_rows_masked(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                              _ptr(v, ctypes.c_uint16), int(dtype), B, H, Nq, Nk, d, float(scale),
                                              int(window_left), int(window_right), int(prefix_len),
                                              _ptr(bh_idx, ctypes.c_int64), _ptr(row_idx, ctypes.c_int64), count,
                                              _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_rows_masked failed (%d)" % rc)
    return o, lse


def attention_fwd_masked_f64(q, k, v, scale: float, window_left: int = -1, window_right: int = -1,
                             prefix_len: int = 0):
    """attention_fwd_masked on float64 inputs q [B,H,Nq,d], k, v [B,H,Nk,d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    o = np.empty((B, H, Nq, d))
    lse = np.empty((B, H, Nq))
    rc = _load().oracle_attention_fwd_masked_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                                 _ptr(v, ctypes.c_double), B, H, Nq, Nk, d, float(scale),
                                                 int(window_left), int(window_right), int(prefix_len),
                                                 _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double))
    if rc:
        raise ValueError("oracle_attention_fwd_masked_f64 failed (%d)" % rc)
    return o, lse


def _bwd_masked_out(B, H, Nq, Nk, d):
    return (np.empty((B, H, Nq, d)), np.empty((B, H, Nk, d)), np.empty((B, H, Nk, d)), np.empty((B, H, Nq)))


def attention_bwd_masked_f64(q, k, v, dout, scale: float, window_left: int = -1, window_right: int = -1,
                             prefix_len: int = 0, threads: int = 0):
    """Gradients (dQ, dK, dV, D) of the masked forward for upstream dout, float64 inputs."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv, delta = _bwd_masked_out(B, H, Nq, Nk, d)
    rc = _load().oracle_attention_bwd_masked_f64(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                                                 _ptr(v, ctypes.c_double), _ptr(dout, ctypes.c_double), B, H, Nq, Nk,
                                                 d, float(scale), int(window_left), int(window_right),
                                                 int(prefix_len), _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                                 _ptr(dv, ctypes.c_double), _ptr(delta, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_bwd_masked_f64 failed (%d)" % rc)
    return dq, dk, dv, delta


def attention_bwd_masked(q, k, v, dout, dtype: int, scale: float, window_left: int = -1, window_right: int = -1,
                         prefix_len: int = 0, threads: int = 0):
    """Masked-backward gradients from 16-bit bit patterns (q, dout [B,H,Nq,d]; k, v [B,H,Nk,d]), float64."""
    q, k, v, dout = _bits(q), _bits(k), _bits(v), _bits(dout)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    dq, dk, dv, delta = _bwd_masked_out(B, H, Nq, Nk, d)
    rc = _load().oracle_attention_bwd_masked(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
                                             _ptr(v, ctypes.c_uint16), _ptr(dout, ctypes.c_uint16), int(dtype), B, H,
                                             Nq, Nk, d, float(scale), int(window_left), int(window_right),
                                             int(prefix_len), _ptr(dq, ctypes.c_double), _ptr(dk, ctypes.c_double),
                                             _ptr(dv, ctypes.c_double), _ptr(delta, ctypes.c_double), int(threads))
    if rc:
        raise ValueError("oracle_attention_bwd_masked failed (%d)" % rc)
    return dq, dk, dv, delta
