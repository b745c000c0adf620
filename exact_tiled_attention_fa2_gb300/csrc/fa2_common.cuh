// fa2_common.cuh -- device helpers shared by the forward kernels: bounded
// mbarrier waits that report to the device status word instead of hanging,
// 16-bit packing, the hi/lo split rule for bf16 P, and the per-tile context.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fa2_internal.h"
#include "sm103_ptx.cuh"

namespace fa2 {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s: far above any legitimate intra-CTA wait

enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaQ = 2,
  kSiteMmaK = 3,
  kSiteMmaP = 4,
  kSiteMmaV = 5,
  kSiteMmaO = 6,
  kSiteSoftmaxS = 7,
  kSiteSoftmaxO = 8,
  kSiteEpilogueO = 9,
  kSiteDrain = 10,
  kSiteSelfTest = 11,
  kSiteDecodeFull = 12,
  kSiteDecodeMerge = 13,
};

// Wait for the phase of `bar` with the given parity for at most `limit_ns`;
// give up early if another role of the CTA has already given up.  On
// expiry: raise the CTA's abort flag, record the site in the device status
// word and return false (the caller then abandons its work and returns).
__device__ __forceinline__ bool wait_or_abort_for(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                                  uint32_t* status, uint32_t site, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > limit_ns) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout | (1u << (8 + site)));
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* status, uint32_t site) {
  return wait_or_abort_for(bar, parity, abort_flag, status, site, kWaitLimitNs);
}

// Bounded wait that ignores the abort flag: used to let this CTA's own copies
// and MMAs finish before it releases shared and tensor memory.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout | (1u << (8 + kSiteDrain)));
      return;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t u) {
  if constexpr (BF16) {
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&u);
    return __bfloat1622float2(h);
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&u);
    return __half22float2(h);
  }
}

// Which keys a query row sees: an additive 0 / -inf mask on S in the sense
// of the Flash Attention 2 page, "Causal masking" (Option A), whose tiles
// that the mask removes entirely are skipped.  For a sequence of N_q queries
// and N_k keys, query i is aligned with key i + off, off = N_k - N_q (the
// last query with the last key), and sees key j < N_k iff
//     j < pre_end                       (a prefix every query sees), or
//     i + off - wl <= j <= i + off + wr (a band; wl or wr < 0: unbounded).
// Causal is (wl, wr) = (-1, 0); a window of w keys back is (w, 0).
struct KeyMask {
  int n_k, off, wl, wr, pre_end;

  // First band key of row i, in [0, n_k] (n_k: none).
  __device__ __forceinline__ int row_lo(int i) const {
    if (wl < 0) return 0;
    const long long x = (long long)i + off - wl;
    return (int)(x < 0 ? 0 : (x > n_k ? n_k : x));
  }
  // Last band key of row i, in [-1, n_k - 1] (-1: none).
  __device__ __forceinline__ int row_hi(int i) const {
    if (wr < 0) return n_k - 1;
    const long long x = (long long)i + off + wr;
    return (int)(x < -1 ? -1 : (x > n_k - 1 ? n_k - 1 : x));
  }
  // Keys [lo, end) some row of [first, last] sees; false if none.  Both band
  // ends are non-decreasing in the row, so this is one interval.
  template <bool BAND>
  __device__ __forceinline__ bool tile_range(int first, int last, int& lo, int& end) const {
    int a = BAND ? row_lo(first) : 0, b = row_hi(last);
    if (pre_end > 0) {
      a = 0;
      b = b > pre_end - 1 ? b : pre_end - 1;
    }
    lo = a;
    end = b + 1;
    return b >= a;
  }
};

// Which key tiles of one query tile need no element mask (every valid row
// sees all of the tile), as thresholds on a tile index t counted from some
// origin: t < pre (inside the prefix) or lo <= t < hi (right of the last
// valid row's left band edge, left of the first row's right band edge and
// inside N_k).
struct TileMask {
  int pre, lo, hi;
  __device__ __forceinline__ bool full(int t) const { return t < pre || (t >= lo && t < hi); }
  // The same thresholds counted from tile index `origin` instead.
  __device__ __forceinline__ TileMask from(int origin) const { return TileMask{pre - origin, lo - origin, hi - origin}; }
};

// Thresholds (tile index 0 = keys [0, bc)) for query rows [first, last].
template <bool BAND>
__device__ __forceinline__ TileMask tile_mask(const KeyMask& km, int first, int last, int bc) {
  TileMask t;
  t.pre = km.pre_end / bc;
  t.lo = BAND ? (km.row_lo(last) + bc - 1) / bc : 0;
  t.hi = (km.row_hi(first) + 1) / bc;  // row_hi <= n_k - 1 keeps the tile inside N_k
  return t;
}

// bf16 P is split into P = P_hi + P_lo (two 16-bit PV products) on tiles
// where rows see few keys: tiles the mask cuts (diagonal and band-edge
// tiles) and every tile when all keys fit in two tiles.  bf16 keeps 8
// significant bits, so a lone rounded P term would otherwise move O by up to
// 2^-9 of a value row; the split brings P to ~16 bits there.
template <bool BF16>
__device__ __forceinline__ bool split_tile(bool masked, bool few_keys) {
  if constexpr (!BF16) {
    return false;
  } else {
    return masked || few_keys;
  }
}

// Set to -inf, in place, the scores of the keys of tile [k0, k0 + BC) that
// query row `row` does not see.  BAND: the first visible key may depend on
// the row (a bounded left window or a prefix); otherwise every row sees keys
// [0, row_hi] and one comparison per score suffices.
template <int BC, bool BAND>
__device__ __forceinline__ void mask_scores(uint32_t* sr, const KeyMask& km, int row, int k0) {
  const int c_hi = km.row_hi(row) - k0;
  if constexpr (BAND) {
    const int c_pre = km.pre_end - k0;
    const int c_lo = km.row_lo(row) - k0;
#pragma unroll
    for (int c = 0; c < BC; ++c) {
      const bool vis = (c < c_pre) || (c >= c_lo && c <= c_hi);
      if (!vis) sr[c] = __float_as_uint(-INFINITY);
    }
  } else {
#pragma unroll
    for (int c = 0; c < BC; ++c)
      if (c > c_hi) sr[c] = __float_as_uint(-INFINITY);
  }
}

// Loads one 64-column box of `rows` rows of head h, batch b, whichever rank
// the map has (3-D maps merge batch and head into one coordinate b*H + h;
// the merged coordinate is precomputed by the caller as `hb`).
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap* map, bool merged, int x, int row, int h,
                                              int b, int hb, uint32_t bar) {
  if (merged)
    tma_load_3d(dst, map, x, row, hb, bar);
  else
    tma_load_4d(dst, map, x, row, h, b, bar);
}

// Stores one 64-column box of rows (the map's box height) of head h, batch b
// from shared memory, whichever rank the map has; tracked by a bulk group.
__device__ __forceinline__ void tma_store_rows(const CUtensorMap* map, bool merged, uint32_t src, int x, int row, int h,
                                               int b, int hb) {
  if (merged)
    tma_store_3d(map, src, x, row, hb);
  else
    tma_store_4d(map, src, x, row, h, b);
}

// One (batch, head) slice: where its rows start in the tensors and how long
// it is.  Packed batches read their offsets from cu_q / cu_k.
struct SeqInfo {
  int b, h;            // batch coordinate in the tensors (0 for packed batches) and head
  int n_q, n_k;
  int row0_q, row0_k;  // first row of the sequence in q/o/lse and in k/v
};

// False (and the bad-offsets status bit set) when the offsets of a
// packed sequence are out of range.
__device__ __forceinline__ bool seq_info(const KernelParams& p, int bh, SeqInfo& s) {
  if (p.bh == p.heads) {  // one batch (the host folds mergeable batches into heads)
    s.b = 0;
    s.h = bh;
  } else {
    s.b = bh / p.heads;
    s.h = bh - s.b * p.heads;
  }
  if (!p.cu_q) {
    s.n_q = p.n_q;
    s.n_k = p.n_k;
    s.row0_q = 0;
    s.row0_k = 0;
    return true;
  }
  const int q_a = __ldg(p.cu_q + s.b), q_b = __ldg(p.cu_q + s.b + 1);
  const int k_a = __ldg(p.cu_k + s.b), k_b = __ldg(p.cu_k + s.b + 1);
  const bool ok = 0 <= q_a && q_a <= q_b && q_b <= p.total_q && q_b - q_a <= p.n_q && 0 <= k_a && k_a <= k_b &&
                  k_b <= p.total_k;
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
    return false;
  }
  s.b = 0;
  s.n_q = q_b - q_a;
  s.n_k = k_b - k_a;
  s.row0_q = q_a;
  s.row0_k = k_a;
  return true;
}

__device__ __forceinline__ KeyMask key_mask(const KernelParams& p, const SeqInfo& s) {
  KeyMask km;
  km.n_k = s.n_k;
  km.off = s.n_k - s.n_q;
  km.wl = p.window_left;
  km.wr = p.window_right;
  km.pre_end = p.prefix < s.n_k ? p.prefix : s.n_k;
  return km;
}

// Per-CTA facts the softmax warps need only in masked tiles and in the
// epilogue.  They live in shared memory (written once before the roles
// split) so that they hold no registers through the main loop.
struct CtaFacts {
  SeqInfo seq;
  KeyMask km;
};

// Epilogue store of one output row: O = O~ / l rounded to 16 bits, LSE in
// natural log; a row that sees no key gets O = 0 and LSE = -inf.
template <int D, bool BF16>
__device__ __forceinline__ void store_row(const KernelParams& p, const SeqInfo& s, int row, uint32_t tO, float m_run,
                                          float l_run) {
  const bool empty = !(l_run > 0.f);
  const float inv_l = empty ? 0.f : 1.f / l_run;
  const bool valid = row < s.n_q;
  uint8_t* o_row = reinterpret_cast<uint8_t*>(p.o) +
                   2 * ((long long)s.b * p.o_bs + (long long)s.h * p.o_hs + (long long)(s.row0_q + row) * p.o_rs);
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tO + c, o);
    tmem_ld_wait_x32(o);
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = empty ? 0u : pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
    if (valid) {
      uint4* dst = reinterpret_cast<uint4*>(o_row + c * 2);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    }
  }
  if (valid)
    p.lse[(long long)s.b * p.l_bs + (long long)s.h * p.l_hs + s.row0_q + row] =
        empty ? -INFINITY : (m_run + log2f(l_run)) * 0.6931471805599453f;
}

// Epilogue through shared memory: row r (0..127) of a tile's O = O~ / l,
// rounded to 16 bits, into sO -- D/64 blocks of 128 rows x 128 bytes with the
// 128-byte swizzle (16-byte chunk c of row r at chunk c ^ (r mod 8)), the
// layout a TMA store of 32-row boxes reads -- and its LSE straight to global
// memory.  A row that sees no key gets O = 0 and LSE = -inf.
template <int D, bool BF16>
__device__ __forceinline__ void stage_row(const KernelParams& p, const SeqInfo& s, int row, int r, uint32_t sO,
                                          uint32_t tO, float m_run, float l_run) {
  const bool empty = !(l_run > 0.f);
  const float inv_l = empty ? 0.f : 1.f / l_run;
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tO + c, o);
    tmem_ld_wait_x32(o);
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = empty ? 0u : pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
    const uint32_t row_base = sO + (uint32_t)(c / 64) * (128u * 128u) + (uint32_t)r * 128u;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int chunk = (c % 64) / 8 + i;
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(row_base + (uint32_t)((chunk ^ (r & 7)) * 16)),
                   "r"(packed[4 * i]), "r"(packed[4 * i + 1]), "r"(packed[4 * i + 2]), "r"(packed[4 * i + 3])
                   : "memory");
    }
  }
  if (row < s.n_q)
    p.lse[(long long)s.b * p.l_bs + (long long)s.h * p.l_hs + s.row0_q + row] =
        empty ? -INFINITY : (m_run + log2f(l_run)) * 0.6931471805599453f;
}

// One warp's 32 staged rows (rows 32 quad .. 32 quad + 31 of the tile whose
// first row is q0) to global memory by TMA; rows past the tensor are clipped
// (unpacked batches only: a packed sequence's tail would reach the next one).
// The warp waits until the stores have completed.
template <int D>
__device__ __forceinline__ void store_staged_rows(const CUtensorMap* tm_o, const KernelParams& p, const SeqInfo& s,
                                                  uint32_t sO, int q0, int quad, int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    const bool merged = p.merged_bh != 0;
    const int hb = s.b * p.heads + s.h;
#pragma unroll
    for (int kb = 0; kb < D / 64; ++kb)
      tma_store_rows(tm_o, merged, sO + (uint32_t)kb * (128u * 128u) + (uint32_t)quad * (32u * 128u), kb * 64,
                     s.row0_q + q0 + quad * 32, s.h, s.b, hb);
    bulk_commit_group();
    // the staging must outlive only TMA's read of it: the writes to global
    // memory complete with the grid
    bulk_wait_read_all();
  }
  __syncwarp();
}

// Rows of a query tile that see no key at all: O = 0, LSE = -inf, without
// touching tensor memory.
template <int D>
__device__ __forceinline__ void store_empty_row(const KernelParams& p, const SeqInfo& s, int row) {
  if (row >= s.n_q) return;
  uint8_t* o_row = reinterpret_cast<uint8_t*>(p.o) +
                   2 * ((long long)s.b * p.o_bs + (long long)s.h * p.o_hs + (long long)(s.row0_q + row) * p.o_rs);
#pragma unroll
  for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(o_row + c * 2) = make_uint4(0u, 0u, 0u, 0u);
  p.lse[(long long)s.b * p.l_bs + (long long)s.h * p.l_hs + s.row0_q + row] = -INFINITY;
}

// Split-key mode: a row's partial over one key chunk -- O~ (unnormalised,
// read from TMEM columns tO.. when `have`, else zeros), m (exp2 domain) and
// l -- into workspace slot (bh * n_q + row) * splits + split, the layout the
// decode merge kernel reads.  Every lane of the warp takes part in the TMEM
// loads (`have` is the same for the whole warp); rows past the sequence store
// nothing.
template <int D>
__device__ __forceinline__ void store_partial_row(const KernelParams& p, int bh, int split, int row, int n_q,
                                                  uint32_t tO, float m, float l, bool have) {
  const bool live = row < n_q;
  const size_t slot = ((size_t)bh * (size_t)p.n_q + (size_t)row) * (size_t)p.splits + (size_t)split;
  float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * D);
#pragma unroll 1
  for (int c = 0; c < D; c += 32) {
    uint32_t o[32];
    if (have) {
      tmem_ld_32x32b_x32(tO + c, o);
      tmem_ld_wait_x32(o);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) o[i] = 0u;
    }
    if (live) {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        dst[c / 4 + i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                     __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
    }
  }
  if (live) {
    p.ws_ml[slot * 2] = m;
    p.ws_ml[slot * 2 + 1] = l;
  }
}

// Order of work units over a 1-D grid of (B*H) x units blocks.  Heads go in
// groups of `group`; inside a group the units run from the last (the one
// with the most key tiles under a causal mask) to the first, heads
// interleaved.  So the CTAs resident at a time share the K/V of about
// kHeadGroup heads in L2, and causal work is launched longest first within
// each group, whose short tail overlaps the next group's long units.
// Forward kernels (128-row units, two CTAs per SM): measured against 4 and 8,
// 16 is 0.2 % faster on B1 H32 N16384 causal and 1 % on B4 H16 N4096 causal;
// 4 loses 7 % on the latter.
constexpr int kHeadGroup = 16;

__device__ __forceinline__ void unit_of_block(int block, int bh_total, int units, int& bh, int& unit,
                                              int group = kHeadGroup) {
  const int full_groups = bh_total / group;
  const int per_group = group * units;
  int g, size, r;
  if (block < full_groups * per_group) {
    g = block / per_group;
    r = block - g * per_group;
    size = group;
  } else {
    g = full_groups;
    r = block - full_groups * per_group;
    size = bh_total - full_groups * group;
  }
  bh = g * group + r % size;
  unit = units - 1 - r / size;
}

// Scratch words packed_unit needs in shared memory.
constexpr int kPackedScanWords = 32;

// Block -> (sequence, head, unit) for packed batches of at most
// kPackedScanSeqs sequences, whose grid holds only the units that exist:
// ceil(n / rows) per (sequence, head), n the sequence's query rows (forward)
// or key rows (backward, `by_keys`).  Sequences whose rows do not overlap hold
// at most total + (rows - 1) * B rows of units between them, which sizes the
// host's grid.  Each thread reads one sequence's offsets, the CTA sums the
// unit counts in packing order, and the thread whose sequence holds this
// block passes its facts on through `scan` (kPackedScanWords ints of shared
// memory).  Inside a sequence the blocks follow unit_of_block over its heads.
// A sequence whose offsets are out of range (the seq_info checks; with
// `by_keys` also more than max_units key tiles) holds no units and sets the
// bad-offsets status bit.  False when this block has no unit; every thread
// returns the same.  `block` (default: this CTA's index) is the grid position
// to place.
template <int THREADS>
__device__ __forceinline__ bool packed_unit(const KernelParams& p, int rows, bool by_keys, int max_units, int group,
                                            int* scan, SeqInfo& s, int& unit, int& units, int block = -1) {
  constexpr int NW = THREADS / 32;
  static_assert(THREADS >= kPackedScanSeqs && NW + 7 <= kPackedScanWords, "packed scan");
  const int nseq = p.bh / p.heads;
  const int i = (int)threadIdx.x, lane = i & 31, w = i >> 5;
  int q_a = 0, q_b = 0, k_a = 0, k_b = 0, cnt = 0;
  if (i < nseq) {
    q_a = __ldg(p.cu_q + i);
    q_b = __ldg(p.cu_q + i + 1);
    k_a = __ldg(p.cu_k + i);
    k_b = __ldg(p.cu_k + i + 1);
    bool ok = 0 <= q_a && q_a <= q_b && q_b <= p.total_q && q_b - q_a <= p.n_q && 0 <= k_a && k_a <= k_b &&
              k_b <= p.total_k;
    if (ok) cnt = ((by_keys ? k_b - k_a : q_b - q_a) + rows - 1) / rows;
    if (ok && by_keys && cnt > max_units) ok = false;
    if (!ok) {
      cnt = 0;
      if (blockIdx.x == 0) atomicOr(p.status, kStatusBadSeqlens);
    }
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (i == 0) scan[NW] = -1;
  if (lane == 31) scan[w] = incl;
  __syncthreads();
  long long start = incl - cnt;
  for (int j = 0; j < w; ++j) start += scan[j];
  const long long blk = block < 0 ? (long long)blockIdx.x : (long long)block;
  if (cnt > 0 && blk >= start * p.heads && blk < (start + cnt) * p.heads) {
    scan[NW] = i;
    scan[NW + 1] = (int)(blk - start * p.heads);
    scan[NW + 2] = cnt;
    scan[NW + 3] = q_a;
    scan[NW + 4] = q_b;
    scan[NW + 5] = k_a;
    scan[NW + 6] = k_b;
  }
  __syncthreads();
  if (scan[NW] < 0) return false;
  units = scan[NW + 2];
  int h;
  unit_of_block(scan[NW + 1], p.heads, units, h, unit, group);
  s.b = 0;
  s.h = h;
  s.row0_q = scan[NW + 3];
  s.n_q = scan[NW + 4] - s.row0_q;
  s.row0_k = scan[NW + 5];
  s.n_k = scan[NW + 6] - s.row0_k;
  return true;
}

}  // namespace fa2
