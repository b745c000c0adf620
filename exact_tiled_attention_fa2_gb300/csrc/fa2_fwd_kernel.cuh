// fa2_fwd_kernel.cuh -- the exact tiled attention forward kernel for sm_103a.
//
// One CTA owns one tile of BR = 128 query rows of one (batch, head) and
// streams the key/value tiles of that head through shared memory
// (FlashAttention V2 in depth, section 2.2: query tiles outside, key/value
// tiles inside, Q loaded once, O written once).  Per key/value tile j:
//
//   S   = Q_i K_j^T                 tcgen05.mma, fp32 accumulator in TMEM
//   m   = max(m, rowmax(S)),  alpha = 2^(m_old - m),  P = 2^(S*scale*log2e - m)
//   l   = alpha * l + rowsum(P)     online softmax (Flash Attention 2 page,
//                                   inner-loop steps 2-4)
//   O~  = alpha * O~ + P V_j        tcgen05.mma with P read from TMEM
//
// and after the last tile O = O~ / l, LSE = (m + log2 l) * ln 2 (section 3.2,
// deferred normalisation; section 7.1, the stored logsumexp).  Causal tiles
// entirely above the diagonal are never visited (section 5.3); tiles that
// cross it, and the ragged last tile, get -inf on the hidden scores.
//
// Warp roles (192 threads):
//   warp 0      TMA producer: Q once, then K_j / V_j into a 2-stage ring
//   warp 1      TMEM owner and MMA issuer (one thread)
//   warps 2-5   softmax: one thread per query row (TMEM lane), so a row's
//               statistics never leave its thread (section 4.2, split-Q)
//
// Every mbarrier wait is bounded in time; on timeout the CTA records the wait
// site in the device status word, abandons the tile, waits (bounded) for its
// own copies and MMAs in flight, frees its TMEM and returns.
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
};

template <int D_, int BC_>
struct FwdConfig {
  static constexpr int D = D_;
  static constexpr int BR = 128;      // query rows per tile = TMEM lanes = MMA M
  static constexpr int BC = BC_;      // keys per streamed tile = MMA N of S
  static constexpr int STAGES = 2;
  static constexpr int THREADS = 192;
  static constexpr uint32_t Q_BYTES = BR * D * 2;
  static constexpr uint32_t KV_BYTES = BC * D * 2;
  // Shared memory (1024-byte aligned regions; each 64-column block of a tile
  // is rows x 128 B in the TMA 128-byte-swizzle layout)
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr uint32_t NUM_BARS = 16;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 1024;  // + slack to align the base
  // Tensor memory columns: S (fp32, BC columns; P overwrites its first BC/2
  // columns as packed 16-bit pairs, and P's low part the next BC/2), then O~.
  static constexpr uint32_t TMEM_S = 0;
  static constexpr uint32_t TMEM_O = 128;
  static constexpr uint32_t TMEM_COLS = (TMEM_O + D <= 256) ? 256 : 512;
  static_assert(D == 64 || D == 128 || D == 256, "head dim");
  static_assert(BC == 64 || BC == 128, "key tile");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Barrier slots
enum : int {
  BAR_Q = 0,
  BAR_KFULL = 1,    // + stage
  BAR_VFULL = 3,    // + stage
  BAR_KVEMPTY = 5,  // + stage
  BAR_S = 7,
  BAR_P = 8,
  BAR_O = 9,
  BAR_EXIT = 10,
};

__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              uint32_t* status, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1;
        atomicOr(status, kStatusTimeout | (site << 8));
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag: used to let this CTA's own copies
// and MMAs finish before it releases shared and tensor memory.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, uint32_t* status) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, kStatusTimeout | (kSiteDrain << 8));
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

struct TileCtx {
  uint32_t bar0;       // shared address of barrier 0
  uint32_t sQ, sK, sV; // shared addresses of the tiles
  uint32_t tmem;       // TMEM base (lane 0, first allocated column)
  volatile int* abort_flag;
  uint32_t* status;
  int bh, q0, n, nkv;
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

template <class C>
__device__ __forceinline__ void run_producer(const TileCtx& t, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_v) {
  mbar_arrive_expect_tx(t.bar(BAR_Q), C::Q_BYTES);
  for (int kb = 0; kb < C::D / 64; ++kb)
    tma_load_3d(t.sQ + kb * (C::BR * 128), tm_q, kb * 64, t.q0, t.bh, t.bar(BAR_Q));
  int last_use[C::STAGES];
  for (int s = 0; s < C::STAGES; ++s) last_use[s] = -1;
  for (int j = 0; j < t.nkv; ++j) {
    const int s = j % C::STAGES;
    const int u = j / C::STAGES;
    if (u > 0 && !wait_or_abort(t.bar(BAR_KVEMPTY + s), (u - 1) & 1, t.abort_flag, t.status, kSiteProducerEmpty))
      break;
    const uint32_t k_dst = t.sK + s * C::KV_BYTES;
    const uint32_t v_dst = t.sV + s * C::KV_BYTES;
    mbar_arrive_expect_tx(t.bar(BAR_KFULL + s), C::KV_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_3d(k_dst + kb * (C::BC * 128), tm_k, kb * 64, j * C::BC, t.bh, t.bar(BAR_KFULL + s));
    mbar_arrive_expect_tx(t.bar(BAR_VFULL + s), C::KV_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_3d(v_dst + kb * (C::BC * 128), tm_v, kb * 64, j * C::BC, t.bh, t.bar(BAR_VFULL + s));
    last_use[s] = u;
  }
  // Own copies in flight land before the CTA may exit.
  wait_drain(t.bar(BAR_Q), 0, t.status);
  for (int s = 0; s < C::STAGES; ++s) {
    if (last_use[s] >= 0) {
      wait_drain(t.bar(BAR_KFULL + s), last_use[s] & 1, t.status);
      wait_drain(t.bar(BAR_VFULL + s), last_use[s] & 1, t.status);
    }
  }
}

template <class C, bool BF16, bool CAUSAL>
__device__ __forceinline__ void run_mma(const TileCtx& t) {
  constexpr uint32_t idesc_qk = make_idesc_f16(C::BR, C::BC, BF16, false, false);
  constexpr uint32_t idesc_pv = make_idesc_f16(C::BR, C::D, BF16, false, true);  // V tile is MN-major
  const uint32_t tS = t.tmem + C::TMEM_S;
  const uint32_t tO = t.tmem + C::TMEM_O;
  if (wait_or_abort(t.bar(BAR_Q), 0, t.abort_flag, t.status, kSiteMmaQ)) {
    tc_fence_after();
    for (int j = 0; j < t.nkv; ++j) {
      const int s = j % C::STAGES;
      const uint32_t u = (uint32_t)(j / C::STAGES);
      if (!wait_or_abort(t.bar(BAR_KFULL + s), u & 1, t.abort_flag, t.status, kSiteMmaK)) break;
      tc_fence_after();
      const uint32_t k_base = t.sK + s * C::KV_BYTES;
#pragma unroll
      for (int k = 0; k < C::D / 16; ++k) {
        const uint64_t a = make_sdesc_sw128(t.sQ + (k >> 2) * (C::BR * 128) + (k & 3) * 32, 16, 1024);
        const uint64_t b = make_sdesc_sw128(k_base + (k >> 2) * (C::BC * 128) + (k & 3) * 32, 16, 1024);
        umma_ss(tS, a, b, idesc_qk, k > 0 ? 1u : 0u);
      }
      umma_commit(t.bar(BAR_S));
      if (!wait_or_abort(t.bar(BAR_P), (uint32_t)j & 1, t.abort_flag, t.status, kSiteMmaP)) break;
      tc_fence_after();
      if (!wait_or_abort(t.bar(BAR_VFULL + s), u & 1, t.abort_flag, t.status, kSiteMmaV)) break;
      tc_fence_after();
      const uint32_t v_base = t.sV + s * C::KV_BYTES;
      const bool split = split_tile<C, BF16, CAUSAL>(j, t.q0, t.n);
#pragma unroll
      for (int k = 0; k < C::BC / 16; ++k) {
        const uint64_t b = make_sdesc_sw128(v_base + k * (16 * 128), C::BC * 128, 1024);
        umma_ts(tO, tS + k * 8, b, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
        if (split) umma_ts(tO, tS + C::BC / 2 + k * 8, b, idesc_pv, 1u);
      }
      umma_commit(t.bar(BAR_KVEMPTY + s));
      umma_commit(t.bar(BAR_O));
      // The next S overwrites the columns P_j is read from: let PV_j finish first.
      if (j + 1 < t.nkv && !wait_or_abort(t.bar(BAR_O), (uint32_t)j & 1, t.abort_flag, t.status, kSiteMmaO))
        break;
    }
  }
  // Every MMA this thread issued completes before TMEM is released.
  umma_commit(t.bar(BAR_EXIT));
  wait_drain(t.bar(BAR_EXIT), 0, t.status);
}

template <class C, bool BF16, bool CAUSAL>
__device__ __forceinline__ void run_softmax(const TileCtx& t, const KernelParams& p, int warp, int lane) {
  const int quad = warp & 3;                   // TMEM lane quarter this warp may access
  const int r = quad * 32 + lane;              // row within the tile = TMEM lane
  const int row = t.q0 + r;                    // query index within the head
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tS = t.tmem + lane_off + C::TMEM_S;
  const uint32_t tO = t.tmem + lane_off + C::TMEM_O;
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY;  // running max, exp2 domain (scores * scale * log2 e)
  float l_run = 0.f;        // running sum of 2^(s - m_run)
  bool ok = true;
  for (int j = 0; j < t.nkv; ++j) {
    ok = wait_or_abort(t.bar(BAR_S), (uint32_t)j & 1, t.abort_flag, t.status, kSiteSoftmaxS);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    uint32_t sr[C::BC];
#pragma unroll
    for (int c = 0; c < C::BC; c += 32) tmem_ld_32x32b_x32(tS + c, sr + c);
#pragma unroll
    for (int c = 0; c < C::BC; c += 32) tmem_ld_wait_x32(sr + c);
    const int k0 = j * C::BC;
    const bool masked = (k0 + C::BC > t.n) || (CAUSAL && (k0 + C::BC - 1 > t.q0));
    if (masked) {
#pragma unroll
      for (int c = 0; c < C::BC; ++c) {
        const int key = k0 + c;
        if (key >= t.n || (CAUSAL && key > row)) sr[c] = __float_as_uint(-INFINITY);
      }
    }
    float mx = -INFINITY;
#pragma unroll
    for (int c = 0; c < C::BC; ++c) mx = fmaxf(mx, __uint_as_float(sr[c]));
    const float m_new = fmaxf(m_run, mx * sl2);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // a row with nothing visible yet stays at 0
    const float alpha = ex2_approx(m_run - m_use);
    const bool split = split_tile<C, BF16, CAUSAL>(j, t.q0, t.n);
    float sum = 0.f;
    uint32_t ph[C::BC / 2];
    uint32_t pl[C::BC / 2];
#pragma unroll
    for (int c = 0; c < C::BC / 2; ++c) {
      const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), sl2, -m_use));
      const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -m_use));
      sum += p0 + p1;
      ph[c] = pack2<BF16>(p0, p1);
      if (split) {
        const float2 h = unpack2<BF16>(ph[c]);
        pl[c] = pack2<BF16>(p0 - h.x, p1 - h.y);
      }
    }
    l_run = l_run * alpha + sum;
#pragma unroll
    for (int c = 0; c < C::BC / 2; c += 32) tmem_st_32x32b_x32(tS + c, ph + c);
    if (split) {
#pragma unroll
      for (int c = 0; c < C::BC / 2; c += 32) tmem_st_32x32b_x32(tS + C::BC / 2 + c, pl + c);
    }
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      // O~ <- alpha * O~ once the previous PV product has landed
      bool ok2 = wait_or_abort(t.bar(BAR_O), (uint32_t)(j - 1) & 1, t.abort_flag, t.status, kSiteSoftmaxO);
      ok2 = __all_sync(0xffffffffu, ok2);
      if (!ok2) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < C::D; c += 32) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tO + c, o);
        tmem_ld_wait_x32(o);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
        tmem_st_32x32b_x32(tO + c, o);
      }
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(t.bar(BAR_P));
    m_run = m_new;
  }
  if (ok) {
    ok = wait_or_abort(t.bar(BAR_O), (uint32_t)(t.nkv - 1) & 1, t.abort_flag, t.status, kSiteEpilogueO);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) return;
  tc_fence_after();
  const float inv_l = 1.f / l_run;
  uint8_t* o_row = reinterpret_cast<uint8_t*>(p.o) + ((size_t)t.bh * (size_t)t.n + (size_t)row) * (C::D * 2);
#pragma unroll 1
  for (int c = 0; c < C::D; c += 32) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tO + c, o);
    tmem_ld_wait_x32(o);
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
      packed[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv_l, __uint_as_float(o[2 * i + 1]) * inv_l);
    if (row < t.n) {
      uint4* dst = reinterpret_cast<uint4*>(o_row + c * 2);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
    }
  }
  if (row < t.n) p.lse[(size_t)t.bh * (size_t)t.n + (size_t)row] = (m_run + log2f(l_run)) * 0.6931471805599453f;
}

template <int D, int BC, bool BF16, bool CAUSAL>
__global__ void __launch_bounds__(192, 1)
    fa2_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const KernelParams p) {
  using C = FwdConfig<D, BC>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);

  TileCtx t;
  t.bar0 = sbase + C::OFF_BAR;
  t.sQ = sbase + C::OFF_Q;
  t.sK = sbase + C::OFF_K;
  t.sV = sbase + C::OFF_V;
  t.abort_flag = abort_flag;
  t.status = p.status;
  t.n = p.n;
  t.bh = (int)blockIdx.x;
  // causal: the longest query tiles (highest index) are launched first
  const int q_tile = CAUSAL ? (int)(gridDim.y - 1 - blockIdx.y) : (int)blockIdx.y;
  t.q0 = q_tile * C::BR;
  const int kv_end = CAUSAL ? min(t.n, t.q0 + C::BR) : t.n;
  t.nkv = (kv_end + C::BC - 1) / C::BC;

  if (threadIdx.x == 0) {
    mbar_init(t.bar(BAR_Q), 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(t.bar(BAR_KFULL + s), 1);
      mbar_init(t.bar(BAR_VFULL + s), 1);
      mbar_init(t.bar(BAR_KVEMPTY + s), 1);
    }
    mbar_init(t.bar(BAR_S), 1);
    mbar_init(t.bar(BAR_P), 4);  // one arrival per softmax warp
    mbar_init(t.bar(BAR_O), 1);
    mbar_init(t.bar(BAR_EXIT), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  t.tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) run_producer<C>(t, &tm_q, &tm_k, &tm_v);
  } else if (warp == 1) {
    if (lane == 0) run_mma<C, BF16, CAUSAL>(t);
    __syncwarp();
  } else {
    run_softmax<C, BF16, CAUSAL>(t, p, warp, lane);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(t.tmem, C::TMEM_COLS);
  }
}

template <int D, int BC, bool BF16, bool CAUSAL>
int launch_fwd(const LaunchArgs& a) {
  using C = FwdConfig<D, BC>;
  auto kern = fa2_fwd_kernel<D, BC, BF16, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  if (e != cudaSuccess) return (int)e;
  dim3 grid((unsigned)a.p.bh, (unsigned)a.p.num_q_tiles);
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.p);
  return (int)cudaGetLastError();
}

template <int D, int BC>
int launch_fwd_dispatch(const LaunchArgs& a) {
  if (a.bf16) return a.causal ? launch_fwd<D, BC, true, true>(a) : launch_fwd<D, BC, true, false>(a);
  return a.causal ? launch_fwd<D, BC, false, true>(a) : launch_fwd<D, BC, false, false>(a);
}

}  // namespace fa2
