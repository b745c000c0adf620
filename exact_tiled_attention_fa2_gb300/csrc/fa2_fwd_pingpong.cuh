// fa2_fwd_pingpong.cuh -- forward kernel for head dims 64 and 128: two query
// tiles per CTA whose softmax work alternates with the other tile's MMAs.
//
// A CTA owns 256 consecutive query rows of one (batch, head) as two 128-row
// tiles A and B that share every streamed K_j / V_j tile (so K/V are read
// from L2 once per 256 rows).  Tensor memory holds S_A, S_B (fp32, 128
// columns each; P overwrites them as packed 16-bit pairs) and O~_A, O~_B.
// The MMA-issuing thread runs, per key/value tile j,
//
//     O~_A += P_A(j) V_j,   S_A(j+1) = Q_A K_{j+1}^T,
//     O~_B += P_B(j) V_j,   S_B(j+1) = Q_B K_{j+1}^T
//
// so while softmax warpgroup A turns S_A(j+1) into P_A(j+1), the tensor pipe
// works on tile B, and the other way round.  tcgen05 MMAs issued by one
// thread execute in order, which is what lets S_t(j+1) be issued into the
// columns P_t(j) is read from right after O~_t += P_t(j) V_j.
//
// The running maximum is only raised when a tile's maximum exceeds it by
// more than kRescaleLog2 (2^8): otherwise P = 2^(s - m) may reach 2^8, which
// 16-bit P and fp32 l and O~ hold exactly as well, and O~ need not be
// rescaled.  The result is the same exact softmax: every term and l use the
// same m, and LSE = (m + log2 l) ln 2.  (Deferred normalisation taken one
// step further than FlashAttention V2 in depth, section 3.2.)
//
// Warp roles (384 threads = 3 warpgroups): warps 0-3 softmax + epilogue of
// tile A, warps 4-7 of tile B (one thread per row = TMEM lane), warp 8 TMEM
// owner and MMA issuer, warp 9 TMA producer, warps 10-11 idle.  The third
// warpgroup gives registers to the two softmax warpgroups (setmaxnreg):
// 2 x 128 x 200 + 128 x 104 = 384 x 168 registers at launch.
//
// Masks and lengths are run-time (KeyMask): each tile visits only the key
// tiles its rows can see, and the two tiles share one stream of them (their
// ranges overlap or touch); key tiles every row sees skip the element mask.
// The epilogue stages O in the tile's (then free) Q buffer and writes it
// with TMA stores (per-row stores for packed batches).
#pragma once

#include "fa2_common.cuh"

namespace fa2 {

constexpr float kRescaleLog2 = 8.0f;

template <int D_>
struct PingPongConfig {
  static constexpr int D = D_;
  static constexpr int BR = 128;   // rows per query tile (MMA M, TMEM lanes)
  static constexpr int BC = 128;   // keys per streamed tile
  static constexpr int NQ = 2;     // query tiles per CTA
  static constexpr int STAGES = (D == 64) ? 3 : 2;
  static constexpr int THREADS = 384;
  static constexpr int MMA_WARP = 8;
  static constexpr int TMA_WARP = 9;
  static constexpr uint32_t REGS_AT_LAUNCH = 168;   // 65536 / 384, rounded down to a multiple of 8
  static constexpr uint32_t REGS_SOFTMAX = 200;
  static constexpr uint32_t REGS_OTHER = 104;
  static_assert(2 * 128 * REGS_SOFTMAX + 128 * REGS_OTHER <= THREADS * REGS_AT_LAUNCH, "register split");
  static constexpr uint32_t Q_BYTES = BR * D * 2;
  static constexpr uint32_t KV_BYTES = BC * D * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + NQ * Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + STAGES * KV_BYTES;
  static constexpr uint32_t NUM_BARS = 32;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t MISC_BYTES = 128;  // TMEM address, abort flag, CtaFacts
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;
  static constexpr uint32_t TMEM_S = 0;     // + 128 * tile
  static constexpr uint32_t TMEM_O = 256;   // + D * tile
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(D == 64 || D == 128, "ping-pong kernel: head dim 64 or 128");
  static_assert(TMEM_O + NQ * D <= TMEM_COLS, "tensor memory");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

enum : int {
  PB_Q = 0,         // + tile
  PB_KFULL = 2,     // + stage (<= 4 stages)
  PB_VFULL = 6,     // + stage
  PB_KVEMPTY = 10,  // + stage
  PB_S = 14,        // + tile
  PB_P = 16,        // + tile
  PB_O = 18,        // + tile: once, after the tile's last PV product
  PB_EXIT = 20,
};

struct PairCtx {
  uint32_t bar0, sQ, sK, sV, tmem;
  volatile int* abort_flag;
  uint32_t* status;
  SeqInfo seq;
  KeyMask km;
  int kv0;       // first streamed key tile (index within the sequence)
  int nu;        // key tiles streamed through the CTA
  int q0[2];     // first query row of each tile
  int first[2];  // streamed index of each tile's first key tile
  int nkv[2];    // key tiles each tile visits (0: none)
  TileMask tm[2];  // unmasked key tiles of each tile, by streamed index
  bool few_keys; // N_k <= 2 key tiles: every bf16 P is split
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <class C>
// Producer.  `first` = true issues what needs no wait -- the Q tiles and the
// first STAGES key/value tiles -- (the kernel does this before its set-up
// barrier, so the loads fly while TMEM is allocated); `first` = false issues
// the rest and then waits for every load in flight to land.
__device__ __forceinline__ void pp_producer(const PairCtx& t, const KernelParams& p, const CUtensorMap* tm_q,
                                            const CUtensorMap* tm_k, const CUtensorMap* tm_v, bool first) {
  const int h = t.seq.h, b = t.seq.b, hb = b * p.heads + h;
  const bool merged = p.merged_bh != 0;
  if (first) {
    for (int q = 0; q < C::NQ; ++q) {
      if (t.nkv[q] == 0) continue;
      mbar_arrive_expect_tx(t.bar(PB_Q + q), C::Q_BYTES);
      for (int kb = 0; kb < C::D / 64; ++kb)
        tma_load_rows(t.sQ + q * C::Q_BYTES + kb * (C::BR * 128), tm_q, merged, kb * 64, t.seq.row0_q + t.q0[q], h,
                      b, hb, t.bar(PB_Q + q));
    }
  }
  int last_use[C::STAGES];
  for (int s = 0; s < C::STAGES; ++s) last_use[s] = s < t.nu ? s / C::STAGES : -1;   // the first pass's stages
  for (int u = first ? 0 : C::STAGES; u < (first ? min(t.nu, C::STAGES) : t.nu); ++u) {
    const int s = u % C::STAGES;
    const int w = u / C::STAGES;
    if (w > 0 && !wait_or_abort(t.bar(PB_KVEMPTY + s), (w - 1) & 1, t.abort_flag, t.status, kSiteProducerEmpty))
      break;
    const int row = t.seq.row0_k + (t.kv0 + u) * C::BC;
    mbar_arrive_expect_tx(t.bar(PB_KFULL + s), C::KV_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sK + s * C::KV_BYTES + kb * (C::BC * 128), tm_k, merged, kb * 64, row, h, b, hb,
                    t.bar(PB_KFULL + s));
    mbar_arrive_expect_tx(t.bar(PB_VFULL + s), C::KV_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sV + s * C::KV_BYTES + kb * (C::BC * 128), tm_v, merged, kb * 64, row, h, b, hb,
                    t.bar(PB_VFULL + s));
    last_use[s] = w;
  }
  if (first) return;
  for (int q = 0; q < C::NQ; ++q)
    if (t.nkv[q] > 0) wait_drain(t.bar(PB_Q + q), 0, t.status);
  for (int s = 0; s < C::STAGES; ++s) {
    if (last_use[s] >= 0) {
      wait_drain(t.bar(PB_KFULL + s), last_use[s] & 1, t.status);
      wait_drain(t.bar(PB_VFULL + s), last_use[s] & 1, t.status);
    }
  }
}

// Descriptors are built once and advanced by adding (byte offset >> 4) to the
// start-address field: every tile sits below 256 KB of shared memory, so the
// 14-bit field never carries into the next one.
template <class C>
__device__ __forceinline__ constexpr uint64_t kmajor_step(int k, int rows) {
  return (uint64_t)(((k >> 2) * (rows * 128) + (k & 3) * 32) >> 4);
}

template <class C, bool BF16, bool BAND>
__device__ __forceinline__ void pp_mma(const PairCtx& t) {
  constexpr uint32_t idesc_qk = make_idesc_f16(C::BR, C::BC, BF16, false, false);
  constexpr uint32_t idesc_pv = make_idesc_f16(C::BR, C::D, BF16, false, true);
  const uint64_t dq0 = make_sdesc_sw128(t.sQ, 16, 1024);
  const uint64_t dk0 = make_sdesc_sw128(t.sK, 16, 1024);
  const uint64_t dv0 = make_sdesc_sw128(t.sV, C::BC * 128, 1024);
  bool ok = true;
  auto issue_s = [&](int q, int u) {
    const uint64_t a0 = dq0 + (uint64_t)((q * C::Q_BYTES) >> 4);
    const uint64_t b0 = dk0 + (uint64_t)(((u % C::STAGES) * C::KV_BYTES) >> 4);
    const uint32_t tS = t.tmem + C::TMEM_S + 128 * q;
#pragma unroll
    for (int k = 0; k < C::D / 16; ++k)
      umma_ss(tS, a0 + kmajor_step<C>(k, C::BR), b0 + kmajor_step<C>(k, C::BC), idesc_qk, k > 0 ? 1u : 0u);
    umma_commit(t.bar(PB_S + q));
  };
  auto issue_pv = [&](int q, int u) {
    const uint64_t b0 = dv0 + (uint64_t)(((u % C::STAGES) * C::KV_BYTES) >> 4);
    const uint32_t tS = t.tmem + C::TMEM_S + 128 * q;
    const uint32_t tO = t.tmem + C::TMEM_O + C::D * q;
    const int jj = BAND ? u - t.first[q] : u;
    if (split_tile<BF16>(!t.tm[q].full(u), t.few_keys)) {
#pragma unroll
      for (int k = 0; k < C::BC / 16; ++k) {
        const uint64_t b = b0 + (uint64_t)((k * 16 * 128) >> 4);
        umma_ts(tO, tS + k * 8, b, idesc_pv, (jj > 0 || k > 0) ? 1u : 0u);
        umma_ts(tO, tS + C::BC / 2 + k * 8, b, idesc_pv, 1u);
      }
    } else {
#pragma unroll
      for (int k = 0; k < C::BC / 16; ++k)
        umma_ts(tO, tS + k * 8, b0 + (uint64_t)((k * 16 * 128) >> 4), idesc_pv, (jj > 0 || k > 0) ? 1u : 0u);
    }
    if (jj + 1 == t.nkv[q]) umma_commit(t.bar(PB_O + q));
  };
#pragma unroll
  for (int q = 0; q < C::NQ; ++q)
    if (ok && t.nkv[q] > 0) ok = wait_or_abort(t.bar(PB_Q + q), 0, t.abort_flag, t.status, kSiteMmaQ);
  if (ok && t.nu > 0) ok = wait_or_abort(t.bar(PB_KFULL), 0, t.abort_flag, t.status, kSiteMmaK);
  if (ok) {
    tc_fence_after();
#pragma unroll
    for (int q = 0; q < C::NQ; ++q)
      if (t.nkv[q] > 0 && t.first[q] == 0) issue_s(q, 0);
    // Per streamed tile u: O~_A += P_A V_u, S_A(u+1); O~_B += P_B V_u, S_B(u+1),
    // each product only for the tiles whose key range holds that tile.  Every
    // u lies in some tile's range (the ranges are made contiguous at set-up),
    // so both loads of stage u are waited for before it is handed back.
    // Without BAND every range starts at streamed tile 0 (first == 0), and
    // the loop needs no branch for a tile that starts later: this loop body
    // is the MMA thread's hot code, and its size shows in the step time.
    for (int u = 0; u < t.nu && ok; ++u) {
      const int s = u % C::STAGES;
      const int s1 = (u + 1) % C::STAGES;
      bool have_v = false, have_k = false;
#pragma unroll
      for (int q = 0; q < C::NQ; ++q) {
        if (!ok) continue;
        const int jj = BAND ? u - t.first[q] : u;
        if (BAND && jj == -1) {  // tile q starts at the next streamed tile: its first S product
          if (!have_k) {
            ok = wait_or_abort(t.bar(PB_KFULL + s1), (uint32_t)((u + 1) / C::STAGES) & 1, t.abort_flag, t.status,
                               kSiteMmaK);
            have_k = true;
            if (!ok) continue;
            tc_fence_after();
          }
          issue_s(q, u + 1);
          continue;
        }
        if (jj < 0 || jj >= t.nkv[q]) continue;
        ok = wait_or_abort(t.bar(PB_P + q), (uint32_t)jj & 1, t.abort_flag, t.status, kSiteMmaP);
        if (ok && !have_v) {
          ok = wait_or_abort(t.bar(PB_VFULL + s), (uint32_t)(u / C::STAGES) & 1, t.abort_flag, t.status, kSiteMmaV);
          have_v = true;
        }
        if (!ok) continue;
        tc_fence_after();
        issue_pv(q, u);
        if (jj + 1 < t.nkv[q]) {
          if (!have_k) {
            ok = wait_or_abort(t.bar(PB_KFULL + s1), (uint32_t)((u + 1) / C::STAGES) & 1, t.abort_flag, t.status,
                               kSiteMmaK);
            have_k = true;
            if (!ok) continue;
            tc_fence_after();
          }
          issue_s(q, u + 1);
        }
      }
      if (ok) umma_commit(t.bar(PB_KVEMPTY + s));
    }
  }
  umma_commit(t.bar(PB_EXIT));
  wait_drain(t.bar(PB_EXIT), 0, t.status);
}

// Exponentiate one 32-column chunk of S into packed 16-bit P (and, when
// SPLIT, its low part P - P_hi) and store it to the chunk's TMEM columns.
template <class C, bool BF16, bool SPLIT>
__device__ __forceinline__ void pp_p_chunk(const uint32_t* sr, int ch, uint32_t tS, float2 scale2, float2 neg_m2,
                                           float2& sum0, float2& sum1) {
  uint32_t ph[16];
  uint32_t pl[16];
#pragma unroll
  for (int c = 0; c < 16; ++c) {
    const int col = ch * 32 + 2 * c;
    float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[col]), __uint_as_float(sr[col + 1])), scale2, neg_m2);
    x.x = ex2_approx(x.x);
    x.y = ex2_approx(x.y);
    if (c & 1)
      sum1 = __fadd2_rn(sum1, x);
    else
      sum0 = __fadd2_rn(sum0, x);
    ph[c] = pack2<BF16>(x.x, x.y);
    if constexpr (SPLIT) {
      const float2 h = unpack2<BF16>(ph[c]);
      pl[c] = pack2<BF16>(x.x - h.x, x.y - h.y);
    }
  }
  tmem_st_32x32b_x16(tS + ch * 16, ph);
  if constexpr (SPLIT) tmem_st_32x32b_x16(tS + C::BC / 2 + ch * 16, pl);
}

template <class C, bool BF16, bool BAND>
__device__ __forceinline__ void pp_softmax(const PairCtx& t, const KernelParams& p, const CtaFacts* facts, int q,
                                           int warp, int lane, const CUtensorMap* tm_o) {
  const int nkv = q ? t.nkv[1] : t.nkv[0];   // selects, not a runtime-indexed local array
  const int q0 = q ? t.q0[1] : t.q0[0];
  const int kt0 = t.kv0 + (q ? t.first[1] : t.first[0]);
  const TileMask tmask = (q ? t.tm[1] : t.tm[0]).from(q ? t.first[1] : t.first[0]);  // by local index j
  const bool few_keys = t.few_keys;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int row = q0 + r;
  if (q0 >= t.seq.n_q) return;
  if (nkv == 0) {
    store_empty_row<C::D>(p, t.seq, row);
    return;
  }
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tS = t.tmem + lane_off + C::TMEM_S + 128 * q;
  const uint32_t tO = t.tmem + lane_off + C::TMEM_O + C::D * q;
  const float sl2 = p.scale_log2;
  float m_run = -INFINITY;  // the maximum the exponentials are taken against (exp2 domain)
  float l_run = 0.f;
  bool ok = true;
  for (int j = 0; j < nkv; ++j) {
    ok = wait_or_abort(t.bar(PB_S + q), (uint32_t)j & 1, t.abort_flag, t.status, kSiteSoftmaxS);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    uint32_t sr[C::BC];
#pragma unroll
    for (int c = 0; c < C::BC; c += 32) tmem_ld_32x32b_x32(tS + c, sr + c);
#pragma unroll
    for (int c = 0; c < C::BC; c += 32) tmem_ld_wait_x32(sr + c);
    const bool masked = !tmask.full(j);
    if (masked) mask_scores<C::BC, BAND>(sr, facts->km, row, (kt0 + j) * C::BC);
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int c = 0; c < C::BC; c += 8) {
      mx0 = fmax3(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
      mx1 = fmax3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
      mx2 = fmax3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
      mx3 = fmax3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
    }
    const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
    const bool raise = m_tile > m_run + kRescaleLog2;   // false when both are -inf
    const float m_new = raise ? m_tile : m_run;
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = raise ? ex2_approx(m_run - m_use) : 1.f;
    const bool split = split_tile<BF16>(masked, few_keys);
    const float2 scale2 = make_float2(sl2, sl2);
    const float2 neg_m2 = make_float2(-m_use, -m_use);
    float2 sum0 = make_float2(0.f, 0.f), sum1 = make_float2(0.f, 0.f);
    // P in 32-column chunks (S is already in registers, so overwriting it is safe)
    if (split) {
#pragma unroll
      for (int ch = 0; ch < C::BC / 32; ++ch) pp_p_chunk<C, BF16, true>(sr, ch, tS, scale2, neg_m2, sum0, sum1);
    } else {
#pragma unroll
      for (int ch = 0; ch < C::BC / 32; ++ch) pp_p_chunk<C, BF16, false>(sr, ch, tS, scale2, neg_m2, sum0, sum1);
    }
    const float2 sum2 = __fadd2_rn(sum0, sum1);
    l_run = l_run * alpha + (sum2.x + sum2.y);
    // O~ <- alpha O~ when the maximum moved.  O~ already holds PV(j-1): the
    // S(j) commit this thread waited on was issued after it, and a commit
    // completes only when every earlier MMA of its issuing thread has.
    if (j > 0 && __any_sync(0xffffffffu, raise)) {
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
    if (lane == 0) mbar_arrive(t.bar(PB_P + q));
    m_run = m_new;
  }
  if (ok) {
    ok = wait_or_abort(t.bar(PB_O + q), 0, t.abort_flag, t.status, kSiteEpilogueO);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) return;
  tc_fence_after();
  if (p.tma_o) {
    // the tile's Q buffer is free: its last S product completed before PB_O
    const uint32_t sO = t.sQ + (uint32_t)q * C::Q_BYTES;
    stage_row<C::D, BF16>(p, facts->seq, row, r, sO, tO, m_run, l_run);
    store_staged_rows<C::D>(tm_o, p, facts->seq, sO, q0, quad, lane);
  } else {
    store_row<C::D, BF16>(p, facts->seq, row, tO, m_run, l_run);
  }
}

// BAND: the first key a query row sees may depend on the row (a bounded left
// window or a prefix), so the two tiles' key ranges may start at different
// key tiles; without it both start at key tile 0.
template <int D, bool BF16, bool BAND>
__global__ void __launch_bounds__(384, 1)
    fa2_fwd_pingpong_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                            const KernelParams p) {
  using C = PingPongConfig<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  CtaFacts* facts = reinterpret_cast<CtaFacts*>(smem + C::OFF_MISC + 16);
  static_assert(16 + sizeof(CtaFacts) <= C::MISC_BYTES, "shared-memory misc area");
  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);

  PairCtx t;
  int bh, pair;
  unit_of_block((int)blockIdx.x, p.bh, p.units, bh, pair);
  // The whole CTA leaves together, before any barrier or TMEM set-up, when
  // its sequence is malformed or shorter than this pair's rows.
  if (!seq_info(p, bh, t.seq)) return;
  if (pair * (C::NQ * C::BR) >= t.seq.n_q) return;
  t.bar0 = sbase + C::OFF_BAR;
  t.sQ = sbase + C::OFF_Q;
  t.sK = sbase + C::OFF_K;
  t.sV = sbase + C::OFF_V;
  t.abort_flag = abort_flag;
  t.status = p.status;
  t.km = key_mask(p, t.seq);
  int lo_tile[C::NQ];
  int kv0 = 0x7fffffff, kv_end = 0;
#pragma unroll
  for (int q = 0; q < C::NQ; ++q) {
    const int q0 = pair * (C::NQ * C::BR) + q * C::BR;
    t.q0[q] = q0;
    t.nkv[q] = 0;
    lo_tile[q] = 0;
    if (q0 < t.seq.n_q) {
      const int last = min(q0 + C::BR, t.seq.n_q) - 1;
      t.tm[q] = tile_mask<BAND>(t.km, q0, last, C::BC);
      int lo, end;
      if (t.km.template tile_range<BAND>(q0, last, lo, end)) {
        lo_tile[q] = lo / C::BC;
        t.nkv[q] = (end + C::BC - 1) / C::BC - lo_tile[q];
        kv0 = min(kv0, lo_tile[q]);
        kv_end = max(kv_end, lo_tile[q] + t.nkv[q]);
      }
    } else {
      t.tm[q] = t.tm[0];
    }
  }
  // The streamed range must have no tile that neither query tile uses.  Both
  // band edges are non-decreasing in the row, so with a tile of each kind the
  // ranges touch or overlap; should they not, tile A is stretched across the
  // gap (the extra tiles are masked out element by element: P = 0 there).
  if (BAND && t.nkv[0] > 0 && t.nkv[1] > 0 && lo_tile[1] > lo_tile[0] + t.nkv[0]) t.nkv[0] = lo_tile[1] - lo_tile[0];
  t.kv0 = kv_end > 0 ? kv0 : 0;
  t.nu = kv_end > 0 ? kv_end - kv0 : 0;
  t.few_keys = t.km.n_k <= 2 * C::BC;
#pragma unroll
  for (int q = 0; q < C::NQ; ++q) {
    t.first[q] = t.nkv[q] > 0 ? lo_tile[q] - t.kv0 : 0;
    t.tm[q] = t.tm[q].from(t.kv0);
  }

  if (warp == C::TMA_WARP && lane == 0) {
    for (int q = 0; q < C::NQ; ++q) {
      mbar_init(t.bar(PB_Q + q), 1);
      mbar_init(t.bar(PB_S + q), 1);
      mbar_init(t.bar(PB_P + q), 4);  // one arrival per softmax warp of the tile
      mbar_init(t.bar(PB_O + q), 1);
    }
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(t.bar(PB_KFULL + s), 1);
      mbar_init(t.bar(PB_VFULL + s), 1);
      mbar_init(t.bar(PB_KVEMPTY + s), 1);
    }
    mbar_init(t.bar(PB_EXIT), 1);
    *abort_flag = 0;
    facts->seq = t.seq;
    facts->km = t.km;
    fence_mbar_init();
    fence_proxy_async_smem();   // the initialised barriers, before this thread's own TMA loads signal them
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    pp_producer<C>(t, p, &tm_q, &tm_k, &tm_v, true);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  t.tmem = *tmem_slot;

  if (warp >= 8) {
    regs_decrease<C::REGS_OTHER>();
    if (warp == C::TMA_WARP) {
      if (lane == 0) pp_producer<C>(t, p, &tm_q, &tm_k, &tm_v, false);
    } else if (warp == C::MMA_WARP) {
      if (lane == 0) pp_mma<C, BF16, BAND>(t);
      __syncwarp();
    }
  } else {
    regs_increase<C::REGS_SOFTMAX>();
    pp_softmax<C, BF16, BAND>(t, p, facts, warp >> 2, warp, lane, &tm_o);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(t.tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool BAND>
int launch_fwd_pingpong(const LaunchArgs& a) {
  using C = PingPongConfig<D>;
  auto kern = fa2_fwd_pingpong_kernel<D, BF16, BAND>;
  static std::atomic<unsigned long long> configured{0};
  const int e = once_per_device(configured, [&]() -> int {
    // The softmax warpgroups' setmaxnreg.inc only completes if the block was
    // launched with the registers the split assumes: refuse to launch otherwise.
    cudaFuncAttributes attr;
    cudaError_t r = cudaFuncGetAttributes(&attr, kern);
    if (r != cudaSuccess) return (int)r;
    if ((uint32_t)attr.numRegs != C::REGS_AT_LAUNCH) return (int)cudaErrorInvalidConfiguration;
    return (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  });
  if (e != 0) return e;
  static_assert(C::NQ * C::BR == 256, "query rows per CTA: tile_geometry(d).cta_rows sizes the grid");
  dim3 grid((unsigned)(a.p.bh * a.p.units));
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
  return (int)cudaGetLastError();
}

template <int D>
int launch_fwd_pingpong_dispatch(const LaunchArgs& a) {
  if (a.band) return a.bf16 ? launch_fwd_pingpong<D, true, true>(a) : launch_fwd_pingpong<D, false, true>(a);
  return a.bf16 ? launch_fwd_pingpong<D, true, false>(a) : launch_fwd_pingpong<D, false, false>(a);
}


}  // namespace fa2
