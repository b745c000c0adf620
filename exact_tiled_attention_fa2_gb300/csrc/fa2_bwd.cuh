// fa2_bwd.cuh -- backward pass of the exact attention forward (head dim 128;
// head dim 64 runs the two-CTA-per-SM variant in fa2_bwd64.cuh, which reuses
// this file's context, helpers and preprocess / convert kernels).
//
// Gradients for an upstream dO (FlashAttention V2 in depth, section 7):
//
//   P   = exp(scale S - L)          S = Q K^T, L the forward logsumexp (7.1)
//   dV  = P^T dO,   dP = dO V^T,    D_i = rowsum(dO_i o O_i)          (7.3)
//   dS  = P o (dP - D),   dQ = scale dS K,   dK = scale dS^T Q
//
// Three kernels:
//   preprocess  D_i = rowsum(dO_i o O_i) in fp32 (its own pass over dO and
//               O, as section 7.3 describes) and zeroes the fp32 dQ accumulator;
//   main        key/value-outer (section 7.2): a CTA owns 128 keys of one
//               (b, h), keeps dK_j and dV_j in tensor memory and walks the
//               query tiles that see those keys; each tile's dQ contribution
//               is staged in shared memory and added to the fp32 accumulator
//               by TMA reduce-add (the accumulation across key tiles, 7.2);
//   convert     dQ accumulator -> 16-bit dQ.
//
// Main kernel, per query tile i (tensor memory holds S^T and dP^T with keys on
// the 128 lanes, so one thread owns one key row):
//   S^T  = K_j Q_i^T              tcgen05.mma, A = K_j, B = Q_i (smem, K-major)
//   dP^T = V_j dO_i^T             tcgen05.mma, A = V_j, B = dO_i
//   P^T, dS^T (16-bit)            elementwise warpgroups, written back to TMEM,
//                                 dS^T also to shared memory
//   dV  += P^T dO_i               A = P^T from TMEM, B = dO_i (MN-major)
//   dK  += dS^T Q_i               A = dS^T from TMEM, B = Q_i (MN-major)
//   dQ_i = dS K_j                 A = dS from smem (MN-major), B = K_j (MN-major),
//                                 into the dP^T columns; each warp copies its 32
//                                 rows out, frees the columns, and TMA adds them
//
// Q_i and dO_i are loaded into separate buffers whose release follows their
// last reader (dK and dV respectively), so the next tile's loads start before
// dQ_i runs.  The tile's MMAs run back to back: issuing the next tile's S^T
// ahead of dK and dQ would need a second Q buffer and a whole tile of dQ
// staging that TMA reads out while the next tile runs (reduce-add drains
// shared memory slowly), which do not fit beside d = 128's tiles.
//
// Warp roles (384 threads): warps 0-3 and 4-7 are two elementwise warpgroups,
// each for 64 of the tile's 128 query columns (and half of the d columns of
// dQ, dK, dV); warp 8 owns TMEM and issues every MMA; warp 9 drives TMA.
// Every mbarrier wait is bounded (fa2_common.cuh), and each barrier is waited
// phase by phase, never more than one phase away from its waiter.
//
// Masks, lengths and layouts are those of the forward pass (KeyMask): a key
// tile visits only the query tiles whose rows see one of its keys -- both
// band edges are non-decreasing in the row, so those rows form one interval
// -- and in a tile some pair of which is hidden, a key row keeps the query
// columns [clo, chi] it is seen by (P = 0 elsewhere).  A key tile no row
// sees stores dK = dV = 0.
#pragma once

#include "fa2_tile.cuh"

namespace fa2 {

template <int D_>
struct BwdConfig {
  static constexpr int D = D_;
  static constexpr int T = 128;                 // rows of a query or key tile
  static constexpr int THREADS = 384;
  static constexpr int MMA_WARP = 8;
  static constexpr int TMA_WARP = 9;
  static constexpr uint32_t TILE_BYTES = T * D * 2;
  static constexpr uint32_t DS_BYTES = T * T * 2;    // dS^T, keys x queries, 16-bit
  static constexpr int QSTAGES = 1;    // Q_i buffers
  static constexpr int DOSTAGES = 1;   // dO_i buffers
  static constexpr uint32_t DQ_BOX_BYTES = 32 * 32 * 4;       // a 32 x 32 fp32 box (one TMA reduce-add)
  static constexpr uint32_t DQ_WARP_BYTES = 32 * (D / 2) * 4;  // a warp's 32 rows x d/2 fp32 dQ columns
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = OFF_K + TILE_BYTES;
  static constexpr uint32_t OFF_Q = OFF_V + TILE_BYTES;             // + stage * TILE_BYTES
  static constexpr uint32_t OFF_DO = OFF_Q + QSTAGES * TILE_BYTES;   // + stage * TILE_BYTES
  static constexpr uint32_t OFF_DS = OFF_DO + DOSTAGES * TILE_BYTES;
  static constexpr uint32_t OFF_DQ = OFF_DS + DS_BYTES;             // + warp * DQ_WARP_BYTES, 32x32 fp32 boxes
  static constexpr uint32_t OFF_BAR = OFF_DQ + 8 * DQ_WARP_BYTES;
  static constexpr uint32_t NUM_BARS = 18;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 4 * kPackedScanWords + 1024;   // misc, scan
  static constexpr uint32_t TMEM_DV = 0;
  static constexpr uint32_t TMEM_DK = 128;
  static constexpr uint32_t TMEM_S = 256;       // S^T, then P^T in its first 32 columns of each half
  static constexpr uint32_t TMEM_DP = 384;      // dP^T, then dS^T, then the dQ_i contribution
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(D == 128, "this backward kernel: head dim 128 (d = 64: fa2_bwd64.cuh)");
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

enum : int {
  BB_KV = 0,
  BB_S = 3,
  BB_DP = 4,
  BB_P = 5,        // P^T, dS^T written (8 warp arrivals)
  BB_DQ = 6,
  BB_DQEMPTY = 7,  // dQ_i read out of TMEM (8 warp arrivals)
  BB_END = 8,
  BB_EXIT = 9,
  BB_Q = 10,        // + stage: Q_i landed
  BB_QEMPTY = 12,   // + stage: the MMAs reading Q_i (S^T, dK) finished
  BB_DO = 14,       // + stage: dO_i landed
  BB_DOEMPTY = 16,  // + stage: the MMAs reading dO_i (dP^T, dV) finished
};

struct BwdCtx {
  uint32_t bar0, sK, sV, sQ, sDO, sDS, tmem;
  volatile int* abort_flag;
  uint32_t* status;
  SeqInfo seq;
  int hb;           // batch * H + head: the merged map coordinate and the workspace slice
  bool merged;      // 3-D maps (batch and head merged) or 4-D
  int j0;           // first key of the tile (within the sequence)
  int i0, niter;    // first query tile visited and how many
  __device__ __forceinline__ uint32_t bar(int i) const { return bar0 + 8u * (uint32_t)i; }
};

template <class C>
// `first` = true issues what needs no wait -- K_j, V_j and the first query
// tile's Q and dO -- (the kernel does this before its set-up barrier, so the
// loads fly while TMEM is allocated) and returns; `first` = false issues the
// rest and then waits for every load in flight to land.
__device__ __forceinline__ void bwd_producer(const BwdCtx& t, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_v, const CUtensorMap* tm_do, bool first) {
  const int h = t.seq.h, b = t.seq.b;
  auto load_q = [&](int it) {
    const int s = it % C::QSTAGES;
    mbar_arrive_expect_tx(t.bar(BB_Q + s), C::TILE_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sQ + s * C::TILE_BYTES + kb * (C::T * 128), tm_q, t.merged, kb * 64,
                    t.seq.row0_q + (t.i0 + it) * C::T, h, b, t.hb, t.bar(BB_Q + s));
  };
  auto load_do = [&](int it) {
    const int s = it % C::DOSTAGES;
    mbar_arrive_expect_tx(t.bar(BB_DO + s), C::TILE_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sDO + s * C::TILE_BYTES + kb * (C::T * 128), tm_do, t.merged, kb * 64,
                    t.seq.row0_q + (t.i0 + it) * C::T, h, b, t.hb, t.bar(BB_DO + s));
  };
  if (first) {
    mbar_arrive_expect_tx(t.bar(BB_KV), 2 * C::TILE_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb) {
      tma_load_rows(t.sK + kb * (C::T * 128), tm_k, t.merged, kb * 64, t.seq.row0_k + t.j0, h, b, t.hb,
                    t.bar(BB_KV));
      tma_load_rows(t.sV + kb * (C::T * 128), tm_v, t.merged, kb * 64, t.seq.row0_k + t.j0, h, b, t.hb,
                    t.bar(BB_KV));
    }
    load_q(0);
    load_do(0);
    return;
  }
  // Q_i into stage i mod QSTAGES once the MMAs of tile i - QSTAGES have read
  // it, then dO_i likewise; in this order Q runs a tile ahead of dO at d = 128
  int loaded_q = 1, loaded_do = 1;   // tile 0's, issued before the set-up barrier
  for (int it = 1; it < t.niter; ++it) {
    const int s = it % C::QSTAGES, u = it / C::QSTAGES;
    if (u > 0 && !wait_or_abort(t.bar(BB_QEMPTY + s), (uint32_t)(u - 1) & 1, t.abort_flag, t.status,
                                kSiteProducerEmpty))
      break;
    load_q(it);
    loaded_q = it + 1;
    const int sd = it % C::DOSTAGES, ud = it / C::DOSTAGES;
    if (ud > 0 && !wait_or_abort(t.bar(BB_DOEMPTY + sd), (uint32_t)(ud - 1) & 1, t.abort_flag, t.status,
                                 kSiteProducerEmpty))
      break;
    load_do(it);
    loaded_do = it + 1;
  }
  // every load in flight lands before the CTA can exit: the last tile of each stage
  wait_drain(t.bar(BB_KV), 0, t.status);
  for (int s = 0; s < C::QSTAGES; ++s) {
    const int last = loaded_q - 1 - ((loaded_q - 1 - s) % C::QSTAGES + C::QSTAGES) % C::QSTAGES;
    if (last >= 0) wait_drain(t.bar(BB_Q + s), (uint32_t)(last / C::QSTAGES) & 1, t.status);
  }
  for (int s = 0; s < C::DOSTAGES; ++s) {
    const int last = loaded_do - 1 - ((loaded_do - 1 - s) % C::DOSTAGES + C::DOSTAGES) % C::DOSTAGES;
    if (last >= 0) wait_drain(t.bar(BB_DO + s), (uint32_t)(last / C::DOSTAGES) & 1, t.status);
  }
}

template <class C, bool BF16>
__device__ __forceinline__ void bwd_mma(const BwdCtx& t) {
  constexpr uint32_t idesc_s = make_idesc_f16(128, C::T, BF16, false, false);     // S^T, dP^T
  constexpr uint32_t idesc_acc = make_idesc_f16(128, C::D, BF16, false, true);    // dV, dK: A in TMEM
  constexpr uint32_t idesc_dq = make_idesc_f16(128, C::D, BF16, true, true);      // dQ: A, B MN-major
  const uint64_t k_kmaj = make_sdesc_sw128(t.sK, 16, 1024);
  const uint64_t v_kmaj = make_sdesc_sw128(t.sV, 16, 1024);
  const uint64_t q_kmaj0 = make_sdesc_sw128(t.sQ, 16, 1024);
  const uint64_t do_kmaj0 = make_sdesc_sw128(t.sDO, 16, 1024);
  const uint64_t q_mn0 = make_sdesc_sw128(t.sQ, C::T * 128, 1024);
  const uint64_t do_mn0 = make_sdesc_sw128(t.sDO, C::T * 128, 1024);
  const uint64_t k_mn = make_sdesc_sw128(t.sK, C::T * 128, 1024);
  const uint64_t ds_mn = make_sdesc_sw128(t.sDS, C::T * 128, 1024);
  const uint32_t tS = t.tmem + C::TMEM_S, tDP = t.tmem + C::TMEM_DP;
  const uint32_t tDV = t.tmem + C::TMEM_DV, tDK = t.tmem + C::TMEM_DK;
  auto issue_s = [&](int q_stage) {   // S^T = K_j Q_i^T for the Q tile in q_stage
    const uint64_t q_kmaj = q_kmaj0 + (uint64_t)((q_stage * C::TILE_BYTES) >> 4);
#pragma unroll
    for (int k = 0; k < C::D / 16; ++k)
      umma_ss(tS, k_kmaj + kmajor_step<C>(k, C::T), q_kmaj + kmajor_step<C>(k, C::T), idesc_s, k > 0 ? 1u : 0u);
    umma_commit(t.bar(BB_S));
  };
  bool ok = wait_or_abort(t.bar(BB_KV), 0, t.abort_flag, t.status, kSiteMmaK);
  // Tile i: S^T_i, dP^T_i, then, once P^T_i and dS^T_i are written, dV, dK, dQ_i
  for (int it = 0; it < t.niter && ok; ++it) {
    const uint32_t ph = (uint32_t)it & 1;
    const int qs = it % C::QSTAGES, ds = it % C::DOSTAGES;
    const uint64_t q_step = (uint64_t)((qs * C::TILE_BYTES) >> 4), do_step = (uint64_t)((ds * C::TILE_BYTES) >> 4);
    const uint64_t do_kmaj = do_kmaj0 + do_step;
    const uint64_t q_mn = q_mn0 + q_step, do_mn = do_mn0 + do_step;
    if (!wait_or_abort(t.bar(BB_Q + qs), (uint32_t)(it / C::QSTAGES) & 1, t.abort_flag, t.status, kSiteMmaQ))
      break;
    tc_fence_after();
    issue_s(qs);
    // dP^T reuses the columns the previous tile's dQ contribution was read from
    if (it > 0 && !wait_or_abort(t.bar(BB_DQEMPTY), ph ^ 1u, t.abort_flag, t.status, kSiteMmaO)) break;
    if (!wait_or_abort(t.bar(BB_DO + ds), (uint32_t)(it / C::DOSTAGES) & 1, t.abort_flag, t.status, kSiteMmaQ)) break;
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < C::D / 16; ++k)
      umma_ss(tDP, v_kmaj + kmajor_step<C>(k, C::T), do_kmaj + kmajor_step<C>(k, C::T), idesc_s, k > 0 ? 1u : 0u);
    umma_commit(t.bar(BB_DP));
    if (!wait_or_abort(t.bar(BB_P), ph, t.abort_flag, t.status, kSiteMmaP)) break;
    tc_fence_after();
    // K = 128 queries in steps of 16: P^T / dS^T of queries 0-63 sit in the
    // first 32 columns of each 64-column half, queries 64-127 in the second half
#pragma unroll
    for (int k = 0; k < C::T / 16; ++k) {
      const uint32_t col = (uint32_t)((k >> 2) * 64 + (k & 3) * 8);
      umma_ts(tDV, tS + col, do_mn + (uint64_t)((k * 16 * 128) >> 4), idesc_acc, (it > 0 || k > 0) ? 1u : 0u);
    }
    umma_commit(t.bar(BB_DOEMPTY + ds));
#pragma unroll
    for (int k = 0; k < C::T / 16; ++k) {
      const uint32_t col = (uint32_t)((k >> 2) * 64 + (k & 3) * 8);
      umma_ts(tDK, tDP + col, q_mn + (uint64_t)((k * 16 * 128) >> 4), idesc_acc, (it > 0 || k > 0) ? 1u : 0u);
    }
    umma_commit(t.bar(BB_QEMPTY + qs));
    // dQ_i = dS K_j into the dP^T columns (the dK products above read dS^T
    // from them first)
#pragma unroll
    for (int k = 0; k < C::T / 16; ++k)
      umma_ss(tDP, ds_mn + (uint64_t)((k * 16 * 128) >> 4), k_mn + (uint64_t)((k * 16 * 128) >> 4), idesc_dq,
              k > 0 ? 1u : 0u);
    umma_commit(t.bar(BB_DQ));
  }
  if (ok) umma_commit(t.bar(BB_END));
  umma_commit(t.bar(BB_EXIT));
  wait_drain(t.bar(BB_EXIT), 0, t.status);
}

// Queries [lo, hi] (within the sequence, clipped to [0, n_q)) that see key
// `key`; lo > hi when none does.
__device__ __forceinline__ void queries_of_key(const KeyMask& km, int n_q, int key, int& lo, int& hi) {
  if (key >= km.n_k) {
    lo = 1;
    hi = 0;
    return;
  }
  long long a = 0, b = n_q - 1;
  if (key >= km.pre_end) {
    if (km.wr >= 0) a = max(a, (long long)key - km.off - km.wr);
    if (km.wl >= 0) b = min(b, (long long)key - km.off + km.wl);
  }
  if (a > b) {
    lo = 1;
    hi = 0;
    return;
  }
  lo = (int)a;
  hi = (int)b;
}

// Query rows [lo, hi] that see some key of [j0, j1] (j0 < n_k <= ...): every
// row when the tile starts inside the prefix, else the rows whose band meets
// the tile, [j0 - off - wr, j1 - off + wl] clipped to [0, n_q); lo > hi when
// there are none.
__device__ __forceinline__ void queries_of_tile(const KeyMask& km, int n_q, int j0, int j1, int& lo, int& hi) {
  long long a = 0, b = n_q - 1;
  if (j0 >= km.pre_end) {
    if (km.wr >= 0) a = max(a, (long long)j0 - km.off - km.wr);
    if (km.wl >= 0) b = min(b, (long long)j1 - km.off + km.wl);
  }
  if (a > b) {
    lo = 1;
    hi = 0;
    return;
  }
  lo = (int)a;
  hi = (int)b;
}

template <class C, bool BF16>
__device__ __forceinline__ void bwd_elementwise(const BwdCtx& t, const BwdParams& p, const KeyMask& km, uint8_t* smem,
                                                int warp, int lane, const CUtensorMap* tm_dq) {
  const KernelParams& f = p.f;
  const int wg = warp >> 2;                // warpgroup: query columns [64 wg, 64 wg + 64)
  const int quad = warp & 3;
  const int r = quad * 32 + lane;          // TMEM lane: key row (S^T, dP^T, dK, dV) or query row (dQ_i)
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tS = t.tmem + lane_off + C::TMEM_S + 64 * wg;
  const uint32_t tDP = t.tmem + lane_off + C::TMEM_DP + 64 * wg;
  uint8_t* ds_row = smem + C::OFF_DS + wg * (C::T * 128) + r * 128;     // this key's row of dS^T, block wg
  uint8_t* dq_stage = smem + C::OFF_DQ + warp * C::DQ_WARP_BYTES;   // this warp's dQ boxes
  const int n_q = t.seq.n_q;
  const int key = t.j0 + r;
  int key_qlo, key_qhi;                    // the queries this key row is seen by
  queries_of_key(km, n_q, key, key_qlo, key_qhi);
  // every (key, query) pair of a 128 x 64 block is visible iff the block's
  // last key is seen from its first query on and its first key up to its last
  int last_qlo, last_qhi, first_qlo, first_qhi;
  queries_of_key(km, n_q, t.j0 + C::T - 1, last_qlo, last_qhi);
  queries_of_key(km, n_q, t.j0, first_qlo, first_qhi);
  const float sl2 = f.scale_log2;
  const float scale = p.scale;
  const long long lse_base = (long long)t.seq.b * f.l_bs + (long long)t.seq.h * f.l_hs + t.seq.row0_q;
  const long long d_base = (long long)t.hb * f.total_q + t.seq.row0_q;
  // dQ of query tile iq (its product runs while the next tile's P^T is
  // computed): read out of TMEM, the columns freed, then added to the fp32
  // accumulator by TMA from shared memory
  auto dq_out = [&](int iq) -> bool {
    bool w = wait_or_abort(t.bar(BB_DQ), (uint32_t)iq & 1, t.abort_flag, t.status, kSiteEpilogueO);
    w = __all_sync(0xffffffffu, w);
    if (!w) return false;
    tc_fence_after();
    // dQ_i rows: lane = query row of tile i; this warpgroup adds d/2 columns.
    // Copy them to registers and free the TMEM columns at once, then stage
    // them in this warp's shared-memory boxes (128-byte swizzle) and let TMA
    // add the boxes to the fp32 accumulator asynchronously (the dQ product
    // has read dS^T: its barrier fired).  Rows past the sequence add zeros
    // (their dS columns are 0).
    uint32_t dq[C::D / 2];
#pragma unroll
    for (int c = 0; c < C::D / 2; c += 32)
      tmem_ld_32x32b_x32(t.tmem + lane_off + C::TMEM_DP + (C::D / 2) * wg + c, dq + c);
#pragma unroll
    for (int c = 0; c < C::D / 2; c += 32) tmem_ld_wait_x32(dq + c);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(t.bar(BB_DQEMPTY));
    // the previous tile's boxes (staged one tile earlier) were read out
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
#pragma unroll
    for (int b = 0; b < C::D / 64; ++b) {
      uint8_t* row = dq_stage + b * C::DQ_BOX_BYTES + lane * 128;
#pragma unroll
      for (int c = 0; c < 8; ++c)
        *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) * 16)) =
            make_uint4(dq[32 * b + 4 * c], dq[32 * b + 4 * c + 1], dq[32 * b + 4 * c + 2], dq[32 * b + 4 * c + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int y = t.seq.row0_q + (t.i0 + iq) * C::T + quad * 32;   // rows past the tensor are clipped
#pragma unroll
      for (int b = 0; b < C::D / 64; ++b)
        tma_reduce_add_3d(tm_dq, smem_u32(dq_stage + b * C::DQ_BOX_BYTES), (C::D / 2) * wg + 32 * b, y, t.hb);
      bulk_commit_group();
    }
    return true;
  };
  bool ok = true;
  for (int it = 0; it < t.niter; ++it) {
    const uint32_t ph = (uint32_t)it & 1;
    const int q0 = (t.i0 + it) * C::T + 64 * wg;   // first query of this warpgroup's columns
    // L (exp2 domain) and D of the 64 queries: lane c holds queries c and
    // c + 32, every lane takes each value by shuffle (warp-local, so no
    // barrier spans warps that might abandon the tile)
    float l_lo, l_hi, d_lo, d_hi;
    {
      const int qa = q0 + lane, qb = q0 + lane + 32;
      l_lo = (qa < n_q) ? f.lse[lse_base + qa] * 1.4426950408889634f : INFINITY;
      l_hi = (qb < n_q) ? f.lse[lse_base + qb] * 1.4426950408889634f : INFINITY;
      d_lo = (qa < n_q) ? p.delta[d_base + qa] : 0.f;
      d_hi = (qb < n_q) ? p.delta[d_base + qb] : 0.f;
    }

    ok = wait_or_abort(t.bar(BB_S), ph, t.abort_flag, t.status, kSiteSoftmaxS);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    uint32_t sr[64];
    tmem_ld_32x32b_x32(tS, sr);
    tmem_ld_32x32b_x32(tS + 32, sr + 32);
    tmem_ld_wait_x32(sr);
    tmem_ld_wait_x32(sr + 32);
    const bool full = last_qlo <= q0 && first_qhi >= q0 + 63 && last_qlo <= last_qhi && first_qlo <= first_qhi;
    float pv[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      const float lq = __shfl_sync(0xffffffffu, c < 32 ? l_lo : l_hi, c & 31);
      pv[c] = ex2_approx(fmaf(__uint_as_float(sr[c]), sl2, -lq));
    }
    // hidden pairs (and rows without keys) give 0; a separate pass that only
    // blocks some pair of which is hidden run
    if (!full) {
      const int clo = key_qlo - q0, chi = key_qhi - q0;   // visible columns of this key row
#pragma unroll
      for (int c = 0; c < 64; ++c)
        if (!(c >= clo && c <= chi)) pv[c] = 0.f;
    }
    uint32_t pk[32];
#pragma unroll
    for (int c = 0; c < 32; ++c) pk[c] = pack2<BF16>(pv[2 * c], pv[2 * c + 1]);
    tmem_st_32x32b_x32(tS, pk);

    ok = wait_or_abort(t.bar(BB_DP), ph, t.abort_flag, t.status, kSiteSoftmaxO);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    uint32_t dr[64];
    tmem_ld_32x32b_x32(tDP, dr);
    tmem_ld_32x32b_x32(tDP + 32, dr + 32);
    tmem_ld_wait_x32(dr);
    tmem_ld_wait_x32(dr + 32);
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float da = __shfl_sync(0xffffffffu, c < 16 ? d_lo : d_hi, (2 * c) & 31);
      const float db = __shfl_sync(0xffffffffu, c < 16 ? d_lo : d_hi, (2 * c + 1) & 31);
      const float a = scale * pv[2 * c] * (__uint_as_float(dr[2 * c]) - da);
      const float b = scale * pv[2 * c + 1] * (__uint_as_float(dr[2 * c + 1]) - db);
      pk[c] = pack2<BF16>(a, b);
    }
    tmem_st_32x32b_x32(tDP, pk);
    // dS^T row to shared memory (128-byte swizzle: 16-byte chunk c of row r
    // at chunk c ^ (r mod 8)), the A operand of the dQ product
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 v = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
      *reinterpret_cast<uint4*>(ds_row + ((c ^ (r & 7)) * 16)) = v;
    }
    fence_proxy_async_smem();
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(t.bar(BB_P));
    if (!dq_out(it)) {
      ok = false;
      break;
    }
  }
  if (lane == 0) bulk_wait_all();   // this warp's reduce-adds performed before the CTA exits
  __syncwarp();
  if (ok && t.niter > 0) {
    ok = wait_or_abort(t.bar(BB_END), 0, t.abort_flag, t.status, kSiteDrain);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) return;
  tc_fence_after();
  // dV_j and dK_j rows (lane = key row): d/2 columns per warpgroup; zero when
  // no query row sees the tile
  const long long col0 = (C::D / 2) * wg;
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const uint32_t base = t.tmem + lane_off + (which ? C::TMEM_DK : C::TMEM_DV) + (C::D / 2) * wg;
    uint8_t* out = reinterpret_cast<uint8_t*>(which ? p.dk : p.dv) +
                   2 * (which ? (long long)t.seq.b * p.k_bs + (long long)t.seq.h * p.k_hs +
                                    (long long)(t.seq.row0_k + key) * p.k_rs + col0
                              : (long long)t.seq.b * p.v_bs + (long long)t.seq.h * p.v_hs +
                                    (long long)(t.seq.row0_k + key) * p.v_rs + col0);
#pragma unroll 1
    for (int c = 0; c < C::D / 2; c += 32) {
      uint32_t pk16[16];
      if (t.niter > 0) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(base + c, o);
        tmem_ld_wait_x32(o);
#pragma unroll
        for (int i = 0; i < 16; ++i) pk16[i] = pack2<BF16>(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]));
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) pk16[i] = 0u;
      }
      if (key < t.seq.n_k) {
        uint4* dst4 = reinterpret_cast<uint4*>(out + c * 2);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst4[i] = make_uint4(pk16[4 * i], pk16[4 * i + 1], pk16[4 * i + 2], pk16[4 * i + 3]);
      }
    }
  }
}

// PACKED: a packed batch whose grid holds only its real key tiles
// (f.packed_units); each CTA finds its sequence and tile from the offsets.
// A template flag, so that the other kernels' code stays as it was.
template <int D, bool BF16, bool PACKED>
__global__ void __launch_bounds__(384, 1)
    fa2_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_dq, const BwdParams p) {
  using C = BwdConfig<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);
  const KernelParams& f = p.f;

  BwdCtx t;
  int bh, unit;
  // heads in groups of 4: a key tile re-streams the Q and dO tiles of every
  // query tile it visits, and 4 heads' worth stay in L2 better than 8 (measured)
  // The whole CTA leaves together, before any set-up, when it has no tile,
  // its sequence is malformed, has more keys than the grid covers, or ends
  // before this tile.
  int units = p.num_k_tiles;
  if constexpr (PACKED) {
    if (!packed_unit<C::THREADS>(f, C::T, true, p.num_k_tiles, 4,
                                 reinterpret_cast<int*>(smem + C::OFF_MISC + 64), t.seq, unit, units))
      return;
  } else {
    unit_of_block((int)blockIdx.x, f.bh, p.num_k_tiles, bh, unit, 4);
    if (!seq_info(f, bh, t.seq)) return;
    if (t.seq.n_k > p.num_k_tiles * C::T) {
      if (threadIdx.x == 0 && unit == 0) atomicOr(f.status, kStatusBadSeqlens);
      return;
    }
  }
  // the key tiles with the most query tiles (the first ones, under a causal
  // mask) start first
  const int jt = units - 1 - unit;
  t.j0 = jt * C::T;
  if (t.j0 >= t.seq.n_k) return;
  const KeyMask km = key_mask(f, t.seq);
  {
    int r_lo, r_hi;
    queries_of_tile(km, t.seq.n_q, t.j0, min(t.j0 + C::T, t.seq.n_k) - 1, r_lo, r_hi);
    t.i0 = r_lo <= r_hi ? r_lo / C::T : 0;
    t.niter = r_lo <= r_hi ? r_hi / C::T - t.i0 + 1 : 0;
  }
  t.hb = t.seq.b * f.heads + t.seq.h;
  t.merged = f.merged_bh != 0;
  t.bar0 = sbase + C::OFF_BAR;
  t.sK = sbase + C::OFF_K;
  t.sV = sbase + C::OFF_V;
  t.sQ = sbase + C::OFF_Q;
  t.sDO = sbase + C::OFF_DO;
  t.sDS = sbase + C::OFF_DS;
  t.abort_flag = abort_flag;
  t.status = f.status;

  if (warp == C::TMA_WARP && lane == 0) {
    mbar_init(t.bar(BB_KV), 1);
    for (int s = 0; s < C::QSTAGES; ++s) {
      mbar_init(t.bar(BB_Q + s), 1);
      mbar_init(t.bar(BB_QEMPTY + s), 1);
    }
    for (int s = 0; s < C::DOSTAGES; ++s) {
      mbar_init(t.bar(BB_DO + s), 1);
      mbar_init(t.bar(BB_DOEMPTY + s), 1);
    }
    mbar_init(t.bar(BB_S), 1);
    mbar_init(t.bar(BB_DP), 1);
    mbar_init(t.bar(BB_P), 8);
    mbar_init(t.bar(BB_DQ), 1);
    mbar_init(t.bar(BB_DQEMPTY), 8);
    mbar_init(t.bar(BB_END), 1);
    mbar_init(t.bar(BB_EXIT), 1);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();   // the initialised barriers, before this thread's own TMA loads signal them
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
    if (t.niter > 0) bwd_producer<C>(t, &tm_q, &tm_k, &tm_v, &tm_do, true);
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
    if (lane == 0 && t.niter > 0) bwd_producer<C>(t, &tm_q, &tm_k, &tm_v, &tm_do, false);
  } else if (warp == C::MMA_WARP) {
    if (lane == 0 && t.niter > 0) bwd_mma<C, BF16>(t);
    __syncwarp();
  } else if (warp < 8) {
    bwd_elementwise<C, BF16>(t, p, km, smem, warp, lane, &tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(t.tmem, C::TMEM_COLS);
  }
}

// D_i = rowsum(dO_i o O_i) in fp32, and the row's fp32 dQ accumulator zeroed,
// for every row of every (batch, head) slice (packed: every row of the
// packed tensors).  D/8 threads per row, 8 elements (16 bytes) each.
template <int D, bool BF16>
__global__ void fa2_bwd_preprocess_kernel(const BwdParams p) {
  constexpr int TPR = D / 8;
  const KernelParams& f = p.f;
  const long long rows = p.slices * f.total_q;
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long row = g / TPR;
  const int part = (int)(g % TPR);
  float acc = 0.f;
  if (row < rows) {
    // a row index fits in 32 bits (2^31 rows of d >= 64 would not fit in memory)
    const int hb = (int)row / f.total_q, i = (int)row - hb * f.total_q;
    const int b = hb / f.heads, h = hb - b * f.heads;
    const long long off = (long long)b * f.o_bs + (long long)h * f.o_hs + (long long)i * f.o_rs + (long long)part * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(f.o) + off);
    const uint4 c = *reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.dout) + off);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 x = unpack2<BF16>(av[k]), y = unpack2<BF16>(cv[k]);
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
    }
    float4* z = reinterpret_cast<float4*>(p.dq_accum + row * D + (long long)part * 8);
    z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int m = TPR / 2; m > 0; m >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, m);
  if (row < rows && part == 0) const_cast<float*>(p.delta)[row] = acc;
}

// 16-bit dQ (q's layout) from the fp32 accumulator, 8 elements per thread.
template <int D, bool BF16>
__global__ void fa2_bwd_dq_convert_kernel(const BwdParams p) {
  const KernelParams& f = p.f;
  const long long n8 = p.slices * f.total_q * (D / 8);
  const long long g = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (g >= n8) return;
  const long long row = g / (D / 8);
  const int part = (int)(g % (D / 8));
  const int hb = (int)row / f.total_q, i = (int)row - hb * f.total_q;   // rows fit in 32 bits
  const int b = hb / f.heads, h = hb - b * f.heads;
  const float4 a = reinterpret_cast<const float4*>(p.dq_accum)[2 * g];
  const float4 c = reinterpret_cast<const float4*>(p.dq_accum)[2 * g + 1];
  uint16_t* dst = reinterpret_cast<uint16_t*>(p.dq) + (long long)b * p.q_bs + (long long)h * p.q_hs +
                  (long long)i * p.q_rs + (long long)part * 8;
  *reinterpret_cast<uint4*>(dst) =
      make_uint4(pack2<BF16>(a.x, a.y), pack2<BF16>(a.z, a.w), pack2<BF16>(c.x, c.y), pack2<BF16>(c.z, c.w));
}

// The main kernel over the grid of key tiles (every key tile of the longest
// sequence per (b, h), or a packed batch's real tiles).
template <int D, bool BF16, bool PACKED>
int launch_bwd_main(const BwdLaunchArgs& a) {
  using C = BwdConfig<D>;
  auto kern = fa2_bwd_kernel<D, BF16, PACKED>;
  static std::atomic<unsigned long long> configured{0};
  const int e = once_per_device(configured, [&]() -> int {
    return (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  });
  if (e != 0) return e;
  const long long blocks = PACKED ? (long long)a.p.f.heads * a.p.f.packed_units : (long long)a.p.f.bh * a.p.num_k_tiles;
  kern<<<(unsigned)blocks, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, a.tm_dq, a.p);
  return (int)cudaGetLastError();
}

template <int D, bool BF16>
int launch_bwd(const BwdLaunchArgs& a) {
  using C = BwdConfig<D>;
  const long long rows = a.p.slices * a.p.f.total_q;   // every row of every (batch, head) slice
  {
    const long long threads = rows * (D / 8);
    fa2_bwd_preprocess_kernel<D, BF16><<<(unsigned)((threads + 255) / 256), 256, 0, a.stream>>>(a.p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  int e = a.p.f.packed_units ? launch_bwd_main<D, BF16, true>(a) : launch_bwd_main<D, BF16, false>(a);
  if (e != 0) return e;
  const long long n8 = rows * (D / 8);
  fa2_bwd_dq_convert_kernel<D, BF16><<<(unsigned)((n8 + 255) / 256), 256, 0, a.stream>>>(a.p);
  return (int)cudaGetLastError();
}

template <int D>
int launch_bwd_dispatch(const BwdLaunchArgs& a) {
  return a.bf16 ? launch_bwd<D, true>(a) : launch_bwd<D, false>(a);
}

}  // namespace fa2
