"""Seeded synthetic inputs shared by the CUDA path's tests/benchmark and the oracle.

This module holds no attention arithmetic: it only draws i.i.d. N(0, 1)
values and rounds them to 16-bit bit patterns, so both sides receive
bit-identical inputs.

Generator: a counter-based splitmix64 (Steele, Lea and Flood, "Fast
splittable pseudorandom number generators", 2014: add the golden-gamma
increment 0x9E3779B97F4A7C15, then the two xor-shift-multiply rounds with
0xBF58476D1CE4E5B9 and 0x94D049BB133111EB and a final xor-shift 31).  The
value at counter c under seed s is mix(s + (c + 1) * gamma).  Element e of
a stream draws two uniforms from counters 2e and 2e + 1, each from the top
24 bits, and forms one normal with the Box-Muller transform
sqrt(-2 ln u1) cos(2 pi u2) (Box and Muller, 1958), evaluated in float64 and
rounded to float32.  Q, K and V are drawn in that order as consecutive
element ranges of one stream over the [B, H, N, d] layout.  The float32
value is then rounded to nearest-even into fp16 or bf16.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

FP16 = 0
BF16 = 1

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def splitmix64(seed: int, counters: np.ndarray) -> np.ndarray:
    """mix(seed + (counter + 1) * gamma) for each counter (uint64 wrap-around)."""
    with np.errstate(over="ignore"):
        c = np.asarray(counters, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (c + np.uint64(1)) * _GAMMA
        return _mix(z)


def _normals_chunk(seed: int, first: int, out: np.ndarray) -> None:
    e = np.arange(first, first + out.size, dtype=np.uint64)
    r1 = splitmix64(seed, e * np.uint64(2))
    r2 = splitmix64(seed, e * np.uint64(2) + np.uint64(1))
    u1 = ((r1 >> np.uint64(40)).astype(np.float64) + 1.0) * (1.0 / 16777216.0)   # (0, 1]
    u2 = (r2 >> np.uint64(40)).astype(np.float64) * (1.0 / 16777216.0)           # [0, 1)
    out[:] = (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)).astype(np.float32)


def normals_f32(seed: int, start: int, count: int) -> np.ndarray:
    """float32 N(0,1) draws for elements [start, start + count) of the stream.

    Chunks are independent (counter-based), so they are filled by a thread
    pool; the result does not depend on the number of threads.
    """
    out = np.empty(count, dtype=np.float32)
    offs = list(range(0, count, _CHUNK))
    if len(offs) <= 1:
        if count:
            _normals_chunk(seed, start, out)
        return out
    workers = min(len(offs), os.cpu_count() or 1, 32)
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(lambda off: _normals_chunk(seed, start + off, out[off:off + _CHUNK]), offs))
    return out


def f32_to_bits(x: np.ndarray, dtype: int) -> np.ndarray:
    """Round float32 to nearest-even fp16 (dtype 0) or bf16 (dtype 1); uint16 bit patterns."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if dtype == FP16:
        return x.astype(np.float16).view(np.uint16)
    if dtype == BF16:
        b = x.view(np.uint32).astype(np.uint64)
        rounded = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
        return rounded.astype(np.uint16)
    raise ValueError("dtype must be 0 (fp16) or 1 (bf16)")


def bits_to_f32(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Exact widening of 16-bit patterns to float32 (for building tensors, not for checking)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == FP16:
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_qkv(B: int, H: int, N: int, d: int, dtype: int, seed: int, q_scale: float = 1.0):
    """Q, K, V as uint16 bit patterns of shape [B, H, N, d].

    ``q_scale`` multiplies the float32 Q draws (in float32) before rounding,
    which sharpens the softmax without changing K or V.
    """
    n = B * H * N * d
    shape = (B, H, N, d)
    q = normals_f32(seed, 0, n)
    if q_scale != 1.0:
        q = (q * np.float32(q_scale)).astype(np.float32)
    q = f32_to_bits(q, dtype).reshape(shape)
    k = f32_to_bits(normals_f32(seed, n, n), dtype).reshape(shape)
    v = f32_to_bits(normals_f32(seed, 2 * n, n), dtype).reshape(shape)
    return q, k, v


@dataclass(frozen=True)
class Workload:
    """One synthetic attention problem: sizes, precision, masking and draw recipe."""
    index: int
    B: int
    H: int
    N: int
    d: int
    dtype: int
    causal: bool
    q_scale: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.d))

    @property
    def name(self) -> str:
        t = "bf16" if self.dtype == BF16 else "fp16"
        extra = " q*%g" % self.q_scale if self.q_scale != 1.0 else ""
        return "B%d H%d N%d d%d %s %s%s" % (self.B, self.H, self.N, self.d, t,
                                            "causal" if self.causal else "non-causal", extra)

    def seed(self, run: int = 0) -> int:
        return 1000 * self.index + run

    def flops(self) -> float:
        """Algorithmic forward FLOPs: 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def algorithmic_bytes(self) -> int:
        """Read Q, K, V once and write O (16-bit) and LSE (fp32) once."""
        return 4 * self.B * self.H * self.N * self.d * 2 + 4 * self.B * self.H * self.N

    def inputs(self, run: int = 0):
        return make_qkv(self.B, self.H, self.N, self.d, self.dtype, self.seed(run), self.q_scale)


def visible_keys(Nq: int, Nk: int, window_left: int = -1, window_right: int = -1, prefix: int = 0) -> np.ndarray:
    """Keys each query row sees under the band / prefix mask (int64 [Nq]).

    Query i is aligned with key i + Nk - Nq and sees key j < Nk iff j < prefix
    or i + off - window_left <= j <= i + off + window_right (-1 = unbounded):
    the count is |[0, prefix) U [lo_i, hi_i]| clipped to [0, Nk).  Used to
    count algorithmic FLOPs (4 d per visible key) of masked problems.
    """
    i = np.arange(Nq, dtype=np.int64)
    off = Nk - Nq
    lo = np.zeros(Nq, np.int64) if window_left < 0 else np.clip(i + off - window_left, 0, Nk)
    hi = np.full(Nq, Nk - 1, np.int64) if window_right < 0 else np.clip(i + off + window_right, -1, Nk - 1)
    band = np.maximum(hi - lo + 1, 0)
    pre = min(max(prefix, 0), Nk)
    overlap = np.where(band > 0, np.maximum(np.minimum(hi + 1, pre) - lo, 0), 0)
    return band + pre - overlap


def union_visible_keys(Nq: int, Nk: int, window_left: int = -1, window_right: int = -1, prefix: int = 0) -> int:
    """Keys that at least one of the Nq query rows sees (same mask as
    visible_keys): the keys whose K and V rows a pass must read.  Counted with
    a difference array over the rows' bands, plus the prefix."""
    i = np.arange(Nq, dtype=np.int64)
    off = Nk - Nq
    lo = np.zeros(Nq, np.int64) if window_left < 0 else np.clip(i + off - window_left, 0, Nk)
    hi = np.full(Nq, Nk - 1, np.int64) if window_right < 0 else np.clip(i + off + window_right, -1, Nk - 1)
    live = hi >= lo
    diff = np.zeros(Nk + 1, np.int64)
    np.add.at(diff, lo[live], 1)
    np.add.at(diff, hi[live] + 1, -1)
    seen = np.cumsum(diff[:Nk]) > 0
    seen[:min(max(prefix, 0), Nk)] = True
    return int(seen.sum())


# The five synthetic workloads: a tiny single-tile case, a short-sequence d=64
# batch, a causal d=128 batch, the long-context causal batch-1 case, and a
# ragged d=256 case with sharpened queries.
WORKLOADS = {
    1: Workload(1, 1, 1, 128, 64, FP16, False),
    2: Workload(2, 8, 16, 2048, 64, FP16, False),
    3: Workload(3, 4, 16, 4096, 128, BF16, True),
    4: Workload(4, 1, 32, 16384, 128, BF16, True),
    5: Workload(5, 2, 8, 3000, 256, FP16, False, q_scale=3.0),
}
