// fa2_fwd_dbuf.cuh -- the forward kernel (head dims 64, 128, 256): one
// 128-row query tile per CTA with two S buffers in tensor memory.
//
// Key/value tiles of B_c = 64 rows stream through separate 2-stage K and V
// rings.  S alternates between two 64-column TMEM buffers, and the
// MMA-issuing thread runs, per key tile j,
//
//     O~ += P(j) V_j,   S(j+2) = Q K_{j+2}^T   (into the buffer P(j) came from)
//
// so the softmax of tile j+1 overlaps those two products.  tcgen05 MMAs
// issued by one thread execute in order, which is what lets S(j+2) follow
// the product reading P(j) from the same columns.  A K stage is released as
// soon as its S product completes and a V stage after its PV product, so the
// next K tile loads while the current PV runs.  At d = 128 the MMA-issuing
// thread waits on one barrier per key tile, P(j): besides the four softmax
// warps, the TMA thread arrives on it once V_j and K_{j+2} have landed, so the
// operand waits are off the MMA thread (each wait there stalls its stream of
// products; see DbufConfig::TMA_GATES_P).  Online softmax with the
// rescaling margin of fa2_tile.cuh: the running max is raised only past 2^8,
// O~ rescaled in place when it is.
//
// Size classes: at d <= 128 a CTA takes 256 TMEM columns (two S buffers +
// O~, and at d = 64 a copy of Q_i) and ~100 KB of shared memory (Q 32 KB at
// d = 128, K and V rings), so two CTAs share an SM: one CTA's set-up, first
// loads and epilogue overlap the other's products, and the two CTAs' MMAs
// interleave on the tensor pipe.  At d = 256 O~ alone takes 256 columns and Q
// 64 KB: one CTA per SM, whose PV products have N = 256.  At d = 64 and 256
// the S products read Q_i from tensor memory (DbufConfig::Q_IN_TMEM).
//
// Warp roles (192 threads): warps 0-3 softmax + epilogue (one thread per
// query row = TMEM lane), warp 4 TMEM owner and MMA issuer, warp 5 TMA.
// Masks and lengths are run-time (KeyMask): the tile visits only the key
// tiles its rows can see; key tiles every row sees skip the element mask.
// The epilogue stages O in the (then free) Q buffer and writes it with TMA
// stores (per-row stores for packed batches).
//
// The same kernel at d = 64 / 128 serves decoding in split-key mode
// (SPLIT; KernelParams::splits > 1): a unit is a (query tile, key chunk) pair,
// the tile's key range is clipped to the chunk, and each row's partial
// (m, l, O~) is written for the decode merge kernel instead of O and LSE.
#pragma once

#include "fa2_tile.cuh"

namespace fa2 {

template <int D_>
struct DbufConfig {
  static constexpr int D = D_;
  static constexpr int BR = 128;
  static constexpr int BC = 64;
  static constexpr int KSTAGES = 2;
  static constexpr int VSTAGES = 2;
  static constexpr int THREADS = 192;
  static constexpr int MMA_WARP = 4;
  static constexpr int TMA_WARP = 5;
  static constexpr uint32_t Q_BYTES = BR * D * 2;
  static constexpr uint32_t KV_BYTES = BC * D * 2;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KSTAGES * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VSTAGES * KV_BYTES;
  static constexpr uint32_t NUM_BARS = 24;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t MISC_BYTES = 128 + 4 * kPackedScanWords;  // TMEM address, abort flag, CtaFacts; scan
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + MISC_BYTES + 1024;
  // Where the columns allow it (d = 64: 224 of 256; d = 256: all 512), the
  // softmax warps copy Q_i once into tensor memory and the S products take it
  // from there as their A operand, reading only K_j from shared memory.
  // Measured on the same GB300: +1.8 % at d = 64 (B8 H16 N2048) and +1.9 % at
  // d = 256 (B2 H8 N3000), same results bit for bit.  At d = 128 two CTAs per
  // SM fill the tensor memory without it.
  static constexpr bool Q_IN_TMEM = (D == 64 || D == 256);
  static constexpr uint32_t TMEM_S = 0;     // + 64 * buffer
  static constexpr uint32_t TMEM_Q = 128;   // Q_i as 16-bit pairs (Q_IN_TMEM)
  static constexpr uint32_t TMEM_O = Q_IN_TMEM ? TMEM_Q + D / 2 : 128;
  static constexpr uint32_t TMEM_COLS = (D == 256) ? 512 : 256;
  static constexpr int CTAS_PER_SM = (D == 256) ? 1 : 2;   // TMEM and shared memory allow two below d = 256
  // The TMA thread, not the MMA thread, checks that V_j and K_{j+2} have landed
  // and says so on P(j).  Measured on the same GB300: d = 128 +1.5-1.8 % (the
  // MMA thread's stream is what limits it there); d = 64 -4.5 % and d = 256
  // -2 %, where the softmax or the single CTA per SM sets the pace and the
  // TMA thread's polling only delays P.
  static constexpr bool TMA_GATES_P = (D == 128);
  static_assert(D == 64 || D == 128 || D == 256, "double-buffered-S kernel: head dim 64, 128 or 256");
  static_assert(TMEM_O + D <= TMEM_COLS, "tensor memory");
  static_assert(CTAS_PER_SM * TMEM_COLS <= 512, "tensor memory per SM");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
  static_assert(CTAS_PER_SM * (SMEM_BYTES + 1024) <= 233472, "shared memory per SM");
};

enum : int {
  DB_Q = 0,
  DB_KFULL = 1,    // + stage
  DB_KEMPTY = 3,   // + stage
  DB_VFULL = 5,    // + stage
  DB_VEMPTY = 7,   // + stage
  DB_S = 9,        // + buffer
  DB_O = 12,       // after every PV product (waited only before a rare O~ rescale)
  DB_EXIT = 13,
  DB_OLAST = 14,   // once, after the last PV product: the epilogue's single-phase wait
  DB_P = 15,       // + buffer.  One per S buffer: S(j+1) is issued before the MMA
                   // thread waits for P(j), so the softmax may finish P(j) and
                   // P(j+1) first; on a single barrier that would put it two
                   // phases ahead of the parity the MMA thread waits for.
                   // Arrivals: the four softmax warps, and with TMA_GATES_P the
                   // TMA thread (V_j and K_{j+2} in shared memory).
  DB_QT = 17,      // Q_IN_TMEM: Q_i copied into tensor memory (four softmax warps)
};

// One query tile's work, shared by the CTA's warp roles.
struct DbufCtx {
  uint32_t bar0, sQ, sK, sV, tmem;
  volatile int* abort_flag;
  uint32_t* status;
  SeqInfo seq;
  KeyMask km;
  int q0;    // first query row of the tile
  int kv0;   // first key tile the tile visits
  int nkv;   // key tiles it visits (0: none)
  int bh, split;  // split-key mode: the (b, h) slice and key chunk of the partials
  TileMask tm;    // unmasked key tiles, by index counted from kv0
  bool few_keys;  // N_k <= 2 key tiles: every bf16 P is split
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

// K_j is needed two products before V_j, so the K and V streams are issued
// independently: whichever ring has a free slot gets the next load.
// `first` = true issues what needs no wait -- Q and the first stage of each
// ring -- (the kernel does this before its set-up barrier, so the loads fly
// while TMEM is allocated) and returns; `first` = false issues the rest and
// then waits for every load in flight to land.
template <class C>
__device__ __forceinline__ void db_producer(const DbufCtx& t, const KernelParams& p, const CUtensorMap* tm_q,
                                            const CUtensorMap* tm_k, const CUtensorMap* tm_v, bool first) {
  const int h = t.seq.h, b = t.seq.b, hb = b * p.heads + h;
  const bool merged = p.merged_bh != 0;
  const int krow0 = t.seq.row0_k + t.kv0 * C::BC;
  const int nk0 = min(t.nkv, C::KSTAGES), nv0 = min(t.nkv, C::VSTAGES);   // loads of the first pass
  if (first) {
    mbar_arrive_expect_tx(t.bar(DB_Q), C::Q_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sQ + kb * (C::BR * 128), tm_q, merged, kb * 64, t.seq.row0_q + t.q0, h, b, hb, t.bar(DB_Q));
    for (int j = 0; j < nk0; ++j) {
      mbar_arrive_expect_tx(t.bar(DB_KFULL + j), C::KV_BYTES);
      for (int kb = 0; kb < C::D / 64; ++kb)
        tma_load_rows(t.sK + j * C::KV_BYTES + kb * (C::BC * 128), tm_k, merged, kb * 64, krow0 + j * C::BC, h, b,
                      hb, t.bar(DB_KFULL + j));
    }
    for (int j = 0; j < nv0; ++j) {
      mbar_arrive_expect_tx(t.bar(DB_VFULL + j), C::KV_BYTES);
      for (int kb = 0; kb < C::D / 64; ++kb)
        tma_load_rows(t.sV + j * C::KV_BYTES + kb * (C::BC * 128), tm_v, merged, kb * 64, krow0 + j * C::BC, h, b,
                      hb, t.bar(DB_VFULL + j));
    }
    return;
  }
  int jk = nk0, jv = nv0;
  int jp = C::TMA_GATES_P ? 0 : t.nkv;   // next key tile whose operands the TMA thread vouches for on P(jp)
  uint64_t idle_since = 0;
  while (jk < t.nkv || jv < t.nkv || jp < t.nkv) {
    bool progressed = false;
    // V_jp and K_{jp+2} issued and landed: arrive on P(jp).  Their barriers are
    // at most one phase ahead: V_{jp+2} and K_{jp+4} load only after products
    // that need P(jp) complete.
    if constexpr (C::TMA_GATES_P) {
      if (jp < jv && (jp + 2 >= t.nkv || jp + 2 < jk) &&
          mbar_try_wait(t.bar(DB_VFULL + jp % C::VSTAGES), (uint32_t)(jp / C::VSTAGES) & 1) &&
          (jp + 2 >= t.nkv ||
           mbar_try_wait(t.bar(DB_KFULL + (jp + 2) % C::KSTAGES), (uint32_t)((jp + 2) / C::KSTAGES) & 1))) {
        mbar_arrive(t.bar(DB_P + (jp & 1)));
        ++jp;
        progressed = true;
      }
    }
    if (jk < t.nkv) {
      const int s = jk % C::KSTAGES, u = jk / C::KSTAGES;
      if (u == 0 || mbar_try_wait(t.bar(DB_KEMPTY + s), (u - 1) & 1)) {
        mbar_arrive_expect_tx(t.bar(DB_KFULL + s), C::KV_BYTES);
        for (int kb = 0; kb < C::D / 64; ++kb)
          tma_load_rows(t.sK + s * C::KV_BYTES + kb * (C::BC * 128), tm_k, merged, kb * 64, krow0 + jk * C::BC, h,
                        b, hb, t.bar(DB_KFULL + s));
        ++jk;
        progressed = true;
      }
    }
    if (jv < t.nkv) {
      const int s = jv % C::VSTAGES, u = jv / C::VSTAGES;
      if (u == 0 || mbar_try_wait(t.bar(DB_VEMPTY + s), (u - 1) & 1)) {
        mbar_arrive_expect_tx(t.bar(DB_VFULL + s), C::KV_BYTES);
        for (int kb = 0; kb < C::D / 64; ++kb)
          tma_load_rows(t.sV + s * C::KV_BYTES + kb * (C::BC * 128), tm_v, merged, kb * 64, krow0 + jv * C::BC, h,
                        b, hb, t.bar(DB_VFULL + s));
        ++jv;
        progressed = true;
      }
    }
    if (progressed) {
      idle_since = 0;
    } else {
      const uint64_t now = global_timer_ns();
      if (idle_since == 0) {
        idle_since = now;
      } else if (*t.abort_flag) {
        break;
      } else if (now - idle_since > kWaitLimitNs) {
        *t.abort_flag = 1;
        atomicOr(t.status, kStatusTimeout | (1u << (8 + kSiteProducerEmpty)));
        break;
      }
    }
  }
  // Own copies in flight land before the CTA may exit.
  wait_drain(t.bar(DB_Q), 0, t.status);
  for (int s = 0; s < C::KSTAGES; ++s) {
    const int last = jk - 1 - ((jk - 1 - s) % C::KSTAGES + C::KSTAGES) % C::KSTAGES;  // last K tile in stage s
    if (last >= 0) wait_drain(t.bar(DB_KFULL + s), (uint32_t)(last / C::KSTAGES) & 1, t.status);
  }
  for (int s = 0; s < C::VSTAGES; ++s) {
    const int last = jv - 1 - ((jv - 1 - s) % C::VSTAGES + C::VSTAGES) % C::VSTAGES;
    if (last >= 0) wait_drain(t.bar(DB_VFULL + s), (uint32_t)(last / C::VSTAGES) & 1, t.status);
  }
}

template <class C, bool BF16>
__device__ __forceinline__ void db_mma(const DbufCtx& t, const KernelParams& p) {
  // S = (+-Q) K^T: a negative scale's sign goes into the product (p.qk_negate)
  const uint32_t idesc_qk = make_idesc_f16(C::BR, C::BC, BF16, false, false) | p.qk_negate;
  constexpr uint32_t idesc_pv = make_idesc_f16(C::BR, C::D, BF16, false, true);
  const uint64_t dq0 = make_sdesc_sw128(t.sQ, 16, 1024);
  const uint64_t dk0 = make_sdesc_sw128(t.sK, 16, 1024);
  const uint64_t dv0 = make_sdesc_sw128(t.sV, C::BC * 128, 1024);
  bool ok = true;
  // with TMA_GATES_P, S(j) for j >= 2 follows a P wait, which covers K_j (see DB_P)
  auto issue_s = [&](int j) -> bool {
    const int sk = j % C::KSTAGES;
    if (!C::TMA_GATES_P || j < 2) {
      if (!wait_or_abort(t.bar(DB_KFULL + sk), (uint32_t)(j / C::KSTAGES) & 1, t.abort_flag, t.status, kSiteMmaK))
        return false;
      tc_fence_after();
    }
    const uint64_t b0 = dk0 + (uint64_t)((sk * C::KV_BYTES) >> 4);
    const uint32_t tS = t.tmem + C::TMEM_S + 64 * (j & 1);
    if constexpr (C::Q_IN_TMEM) {
#pragma unroll
      for (int k = 0; k < C::D / 16; ++k)   // 16 elements of the head dim = 8 columns of Q_i
        umma_ts(tS, t.tmem + C::TMEM_Q + k * 8, b0 + kmajor_step<C>(k, C::BC), idesc_qk, k > 0 ? 1u : 0u);
    } else {
#pragma unroll
      for (int k = 0; k < C::D / 16; ++k)
        umma_ss(tS, dq0 + kmajor_step<C>(k, C::BR), b0 + kmajor_step<C>(k, C::BC), idesc_qk, k > 0 ? 1u : 0u);
    }
    umma_commit(t.bar(DB_S + (j & 1)));
    umma_commit(t.bar(DB_KEMPTY + sk));
    return true;
  };
  if (t.nkv > 0 && wait_or_abort(t.bar(C::Q_IN_TMEM ? DB_QT : DB_Q), 0, t.abort_flag, t.status, kSiteMmaQ)) {
    tc_fence_after();
    ok = issue_s(0);
    if (ok && t.nkv > 1) ok = issue_s(1);
    for (int j = 0; j < t.nkv && ok; ++j) {
      const int sv = j % C::VSTAGES;
      // with TMA_GATES_P, P(j) also stands for V_j and K_{j+2} in shared memory
      ok = wait_or_abort(t.bar(DB_P + (j & 1)), (uint32_t)(j >> 1) & 1, t.abort_flag, t.status, kSiteMmaP);
      if (!C::TMA_GATES_P)
        ok = ok &&
             wait_or_abort(t.bar(DB_VFULL + sv), (uint32_t)(j / C::VSTAGES) & 1, t.abort_flag, t.status, kSiteMmaV);
      if (!ok) break;
      tc_fence_after();
      const uint64_t b0 = dv0 + (uint64_t)((sv * C::KV_BYTES) >> 4);
      const uint32_t tS = t.tmem + C::TMEM_S + 64 * (j & 1);
      const uint32_t tO = t.tmem + C::TMEM_O;
      if (split_tile<BF16>(!t.tm.full(j), t.few_keys)) {
#pragma unroll
        for (int k = 0; k < C::BC / 16; ++k) {
          const uint64_t b = b0 + (uint64_t)((k * 16 * 128) >> 4);
          umma_ts(tO, tS + k * 8, b, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
          umma_ts(tO, tS + C::BC / 2 + k * 8, b, idesc_pv, 1u);
        }
      } else {
#pragma unroll
        for (int k = 0; k < C::BC / 16; ++k)
          umma_ts(tO, tS + k * 8, b0 + (uint64_t)((k * 16 * 128) >> 4), idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(t.bar(DB_O));
      umma_commit(t.bar(DB_VEMPTY + sv));
      if (j + 1 == t.nkv) umma_commit(t.bar(DB_OLAST));
      // S(j+2) reuses the columns P(j) is read from: in-order MMA execution
      // lets it follow the product above directly
      if (j + 2 < t.nkv) ok = issue_s(j + 2);
    }
  }
  umma_commit(t.bar(DB_EXIT));
  wait_drain(t.bar(DB_EXIT), 0, t.status);
}

template <class C, bool BF16, bool BAND, bool SPLIT>
__device__ __forceinline__ void db_softmax(const DbufCtx& t, const KernelParams& p, const CtaFacts* facts, int warp,
                                           int lane, const CUtensorMap* tm_o) {
  const int quad = warp & 3;
  const int r = quad * 32 + lane;
  const int row = t.q0 + r;
  if (t.nkv == 0) {
    if (SPLIT)
      store_partial_row<C::D>(p, t.bh, t.split, row, t.seq.n_q, 0u, -INFINITY, 0.f, false);
    else
      store_empty_row<C::D>(p, t.seq, row);
    return;
  }
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tO = t.tmem + lane_off + C::TMEM_O;
  const float sl2 = p.scale_log2_mag;
  const TileMask tmask = t.tm;
  const bool few_keys = t.few_keys;
  float m_run = -INFINITY;
  float l_run = 0.f;
  bool ok = true;
  if constexpr (C::Q_IN_TMEM) {
    // Row r of Q_i from its 128-byte-swizzled shared-memory blocks (16-byte
    // chunk c of a row stored at chunk c ^ (r & 7)) into TMEM lane r, 64
    // elements = 32 columns per block.  TMA has zero-filled rows past N.
    ok = wait_or_abort(t.bar(DB_Q), 0, t.abort_flag, t.status, kSiteMmaQ);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
#pragma unroll 1
      for (int kb = 0; kb < C::D / 64; ++kb) {
        const uint32_t src = t.sQ + kb * (C::BR * 128) + r * 128;
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 x = lds128(src + ((c ^ (r & 7)) << 4));
          w[4 * c] = x.x;
          w[4 * c + 1] = x.y;
          w[4 * c + 2] = x.z;
          w[4 * c + 3] = x.w;
        }
        tmem_st_32x32b_x32(t.tmem + lane_off + C::TMEM_Q + kb * 32, w);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(t.bar(DB_QT));
    }
  }
  for (int j = 0; ok && j < t.nkv; ++j) {
    const uint32_t tS = t.tmem + lane_off + C::TMEM_S + 64 * (j & 1);
    ok = wait_or_abort(t.bar(DB_S + (j & 1)), (uint32_t)(j >> 1) & 1, t.abort_flag, t.status, kSiteSoftmaxS);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    uint32_t sr[C::BC];
#pragma unroll
    for (int c = 0; c < C::BC; c += 32) tmem_ld_32x32b_x32(tS + c, sr + c);
#pragma unroll
    for (int c = 0; c < C::BC; c += 32) tmem_ld_wait_x32(sr + c);
    const bool masked = !tmask.full(j);
    if (masked) mask_scores<C::BC, BAND>(sr, facts->km, row, (t.kv0 + j) * C::BC);
    float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
    for (int c = 0; c < C::BC; c += 8) {
      mx0 = fmax3(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
      mx1 = fmax3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
      mx2 = fmax3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
      mx3 = fmax3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
    }
    // the largest scaled score (sl2 > 0, so scaling keeps the maximum's place)
    const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * sl2;
    const bool raise = m_tile > m_run + kRescaleLog2;
    const float m_new = raise ? m_tile : m_run;
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = raise ? ex2_approx(m_run - m_use) : 1.f;
    const float2 scale2 = make_float2(sl2, sl2);
    const float2 neg_m2 = make_float2(-m_use, -m_use);
    float2 sum0 = make_float2(0.f, 0.f), sum1 = make_float2(0.f, 0.f);
    if (split_tile<BF16>(masked, few_keys)) {
#pragma unroll
      for (int ch = 0; ch < C::BC / 32; ++ch) softmax_p_chunk<C, BF16, true>(sr, ch, tS, scale2, neg_m2, sum0, sum1);
    } else {
#pragma unroll
      for (int ch = 0; ch < C::BC / 32; ++ch) softmax_p_chunk<C, BF16, false>(sr, ch, tS, scale2, neg_m2, sum0, sum1);
    }
    const float2 sum2 = __fadd2_rn(sum0, sum1);
    l_run = l_run * alpha + (sum2.x + sum2.y);
    if (j > 0 && __any_sync(0xffffffffu, raise)) {
      // S(j) was issued before PV(j-1): wait for that product before rescaling
      // O~.  S(j) completing implies PV(j-2) did, so this barrier is at phase
      // j-1 or j and the parity wait is unambiguous.
      bool ok2 = wait_or_abort(t.bar(DB_O), (uint32_t)(j - 1) & 1, t.abort_flag, t.status, kSiteSoftmaxO);
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
    if (lane == 0) mbar_arrive(t.bar(DB_P + (j & 1)));
    m_run = m_new;
  }
  if (ok) {
    // Not the every-product barrier: S(j+1) is issued before PV(j), so it can
    // still be two phases behind here, where a parity wait would pass early.
    ok = wait_or_abort(t.bar(DB_OLAST), 0, t.abort_flag, t.status, kSiteEpilogueO);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) return;
  tc_fence_after();
  if (SPLIT) {
    store_partial_row<C::D>(p, t.bh, t.split, row, t.seq.n_q, tO, m_run, l_run, true);
  } else if (p.tma_o) {
    // the Q buffer is free: the last S product completed before DB_OLAST
    stage_row<C::D, BF16>(p, facts->seq, row, r, t.sQ, tO, m_run, l_run);
    store_staged_rows<C::D>(tm_o, p, facts->seq, t.sQ, t.q0, quad, lane);
  } else {
    store_row<C::D, BF16>(p, facts->seq, row, tO, m_run, l_run);
  }
}

// BAND: the first key a query row sees may depend on the row (a bounded left
// window or a prefix); it selects the element mask's form.  SPLIT: split-key
// mode (decoding; p.splits > 1), instantiated for the decode path only.
// PACKED: a packed batch whose grid holds only its real tiles
// (p.packed_units); each CTA finds its sequence and tile from the offsets.
// A template flag, so that the other kernels' code stays as it was.
template <int D, bool BF16, bool BAND, bool SPLIT = false, bool PACKED = false>
__global__ void __launch_bounds__(192, DbufConfig<D>::CTAS_PER_SM)
    fa2_fwd_dbuf_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                        const KernelParams p) {
  using C = DbufConfig<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  CtaFacts* facts = reinterpret_cast<CtaFacts*>(smem + C::OFF_MISC + 16);
  static_assert(16 + sizeof(CtaFacts) <= 128, "shared-memory misc area");
  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);

  DbufCtx t;
  int bh, unit;
  static_assert(!(SPLIT && PACKED), "split-key mode runs on the plain grid");
  const int splits = SPLIT ? p.splits : 1;
  if (SPLIT) grid_launch_dependents();   // the decode merge may be scheduled now; it waits for the partials
  // The whole CTA leaves together, before any barrier or TMEM set-up, when
  // it has no tile, its sequence is malformed or shorter than this tile's rows.
  // (The packed kernels keep the plain path behind a run-time test: built
  // that way they measured 8 % faster on packed batches than built without.)
  if (PACKED && p.packed_units) {
    int units;
    if (!packed_unit<C::THREADS>(p, C::BR, false, 0, kHeadGroup,
                                 reinterpret_cast<int*>(smem + C::OFF_MISC + 128), t.seq, unit, units))
      return;
    bh = t.seq.h;   // t.bh serves split-key mode only
  } else {
    unit_of_block((int)blockIdx.x, p.bh, p.units, bh, unit);
    if (!seq_info(p, bh, t.seq)) return;
  }
  const int q_tile = unit / splits;
  t.bh = bh;
  t.split = unit - q_tile * splits;
  if (SPLIT && t.seq.n_k > p.split_base + splits * p.split_chunk) {   // a packed sequence the plan does not cover
    if (threadIdx.x == 0 && t.split == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  t.q0 = q_tile * C::BR;
  if (t.q0 >= t.seq.n_q) return;
  t.bar0 = sbase + C::OFF_BAR;
  t.sQ = sbase + C::OFF_Q;
  t.sK = sbase + C::OFF_K;
  t.sV = sbase + C::OFF_V;
  t.abort_flag = abort_flag;
  t.status = p.status;
  t.km = key_mask(p, t.seq);
  const int last = min(t.q0 + C::BR, t.seq.n_q) - 1;
  int lo, end;
  bool any = t.km.template tile_range<BAND>(t.q0, last, lo, end);
  if (SPLIT && any) {   // the chunk's keys only (chunks are whole key tiles)
    lo = max(lo, p.split_base + t.split * p.split_chunk);
    end = min(end, p.split_base + (t.split + 1) * p.split_chunk);
    any = lo < end;
  }
  if (any) {
    t.kv0 = lo / C::BC;
    t.nkv = (end + C::BC - 1) / C::BC - t.kv0;
  } else {
    t.kv0 = 0;
    t.nkv = 0;
  }
  t.tm = tile_mask<BAND>(t.km, t.q0, last, C::BC).from(t.kv0);
  t.few_keys = t.km.n_k <= 2 * C::BC;

  if (warp == C::TMA_WARP && lane == 0) {
    mbar_init(t.bar(DB_Q), 1);
    for (int s = 0; s < C::KSTAGES; ++s) {
      mbar_init(t.bar(DB_KFULL + s), 1);
      mbar_init(t.bar(DB_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::VSTAGES; ++s) {
      mbar_init(t.bar(DB_VFULL + s), 1);
      mbar_init(t.bar(DB_VEMPTY + s), 1);
    }
    mbar_init(t.bar(DB_S), 1);
    mbar_init(t.bar(DB_S + 1), 1);
    mbar_init(t.bar(DB_P), C::TMA_GATES_P ? 5 : 4);   // one arrival per softmax warp (and the TMA thread)
    mbar_init(t.bar(DB_P + 1), C::TMA_GATES_P ? 5 : 4);
    mbar_init(t.bar(DB_O), 1);
    mbar_init(t.bar(DB_OLAST), 1);
    mbar_init(t.bar(DB_EXIT), 1);
    if (C::Q_IN_TMEM) mbar_init(t.bar(DB_QT), 4);
    *abort_flag = 0;
    facts->seq = t.seq;
    facts->km = t.km;
    fence_mbar_init();
    fence_proxy_async_smem();   // the initialised barriers, before this thread's own TMA loads signal them
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_o);
    if (t.nkv > 0) db_producer<C>(t, p, &tm_q, &tm_k, &tm_v, true);
  }
  if (warp == C::MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  t.tmem = *tmem_slot;

  if (warp == C::TMA_WARP) {
    if (lane == 0 && t.nkv > 0) db_producer<C>(t, p, &tm_q, &tm_k, &tm_v, false);
  } else if (warp == C::MMA_WARP) {
    if (lane == 0) db_mma<C, BF16>(t, p);
    __syncwarp();
  } else {
    db_softmax<C, BF16, BAND, SPLIT>(t, p, facts, warp, lane, &tm_o);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(t.tmem, C::TMEM_COLS);
  }
}

template <int D, bool BF16, bool BAND, bool SPLIT = false, bool PACKED = false>
int launch_fwd_dbuf(const LaunchArgs& a) {
  using C = DbufConfig<D>;
  auto kern = fa2_fwd_dbuf_kernel<D, BF16, BAND, SPLIT, PACKED>;
  static std::atomic<unsigned long long> configured{0};
  const int e = once_per_device(configured, [&]() -> int {
    return (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  });
  if (e != 0) return e;
  static_assert(C::BR == 128, "query rows per CTA: tile_geometry(d).cta_rows sizes the grid");
  dim3 grid((unsigned)(PACKED ? a.p.heads * a.p.packed_units : a.p.bh * a.p.units));
  kern<<<grid, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
  return (int)cudaGetLastError();
}

template <int D>
int launch_fwd_dbuf_dispatch(const LaunchArgs& a) {
  if (a.p.packed_units) {
    if (a.band) return a.bf16 ? launch_fwd_dbuf<D, true, true, false, true>(a) : launch_fwd_dbuf<D, false, true, false, true>(a);
    return a.bf16 ? launch_fwd_dbuf<D, true, false, false, true>(a) : launch_fwd_dbuf<D, false, false, false, true>(a);
  }
  if (a.band) return a.bf16 ? launch_fwd_dbuf<D, true, true>(a) : launch_fwd_dbuf<D, false, true>(a);
  return a.bf16 ? launch_fwd_dbuf<D, true, false>(a) : launch_fwd_dbuf<D, false, false>(a);
}


}  // namespace fa2
