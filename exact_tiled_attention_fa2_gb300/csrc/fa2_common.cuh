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

// A key tile is split into P = P_hi + P_lo (two 16-bit PV products) when the
// input is bf16 and the tile is one where rows see few keys: tiles crossing
// the causal diagonal, or every tile when all keys fit in two tiles.  bf16
// keeps 8 significant bits, so a lone rounded P term would otherwise move O
// by up to 2^-9 of a value row; the split brings P to ~16 bits there.
template <class C, bool BF16, bool CAUSAL>
__device__ __forceinline__ bool split_tile(int j, int q0, int n) {
  if constexpr (!BF16) {
    return false;
  } else {
    const bool diag = CAUSAL && (j * C::BC + C::BC - 1 > q0);
    return diag || (n <= 2 * C::BC);
  }
}

// Order of work units over a 1-D grid of (B*H) x units blocks.  Heads go in
// groups of kHeadGroup; inside a group the units run from the last (the one
// with the most key tiles under a causal mask) to the first, heads
// interleaved.  So the CTAs resident at a time share the K/V of about
// kHeadGroup heads in L2, and causal work is launched longest first within
// each group, whose short tail overlaps the next group's long units.
constexpr int kHeadGroup = 8;

__device__ __forceinline__ void unit_of_block(int block, int bh_total, int units, int& bh, int& unit) {
  const int full_groups = bh_total / kHeadGroup;
  const int per_group = kHeadGroup * units;
  int g, size, r;
  if (block < full_groups * per_group) {
    g = block / per_group;
    r = block - g * per_group;
    size = kHeadGroup;
  } else {
    g = full_groups;
    r = block - full_groups * per_group;
    size = bh_total - full_groups * kHeadGroup;
  }
  bh = g * kHeadGroup + r % size;
  unit = units - 1 - r / size;
}

// Addresses and sizes of one query tile's work, shared by its warp roles.
struct TileCtx {
  uint32_t bar0;       // shared address of barrier 0
  uint32_t sQ, sK, sV; // shared addresses of the tiles
  uint32_t tmem;       // TMEM base (lane 0, first allocated column)
  volatile int* abort_flag;
  uint32_t* status;
  int bh, q0, n, nkv;
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

}  // namespace fa2
