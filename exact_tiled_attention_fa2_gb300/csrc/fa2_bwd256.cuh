// fa2_bwd256.cuh -- backward pass at head dim 256.
//
// The same gradients as fa2_bwd.cuh (FlashAttention V2 in depth, section 7;
// key/value-outer, dQ accumulated across key tiles by TMA reduce-add).  At
// d = 256 the accumulators of 128 keys, dK_j and dV_j, would fill all 512
// columns of tensor memory by themselves, so the output columns are split:
// a CTA owns 128 keys and one half c of the head dimension (columns
// [128 c, 128 c + 128) of dK, dV and dQ); the two halves of a key tile run in
// separate CTAs, each recomputing the tile's S^T and dP^T (products over the
// whole d = 256).  Query tiles have 64 rows, as in fa2_bwd64.cuh, so Q_t and
// dO_t fit twice in shared memory.
//
// TMEM (512 columns): dV_c [0, 128), dK_c [128, 256), S^T [256, 320) then P^T
// in its first 32 columns, dP^T [320, 384) then dS^T, V_j [384, 512) as the A
// operand of dP^T = V_j dO_t^T (keys on the lanes, d/2 columns of 16-bit
// pairs; the elementwise warps load it once).  dQ of a pair of query tiles,
// an M = 128 product dS K_j[:, c], goes into [256, 384) once dV and dK have
// read P^T and dS^T there; the next S^T waits until the elementwise warps have
// read dQ out.
//
// Shared memory: K_j (64 KB; A of S^T, and its half c is B of dQ), two stages
// of Q_t and of dO_t (32 KB each), and the pair's dS^T (two 64-query halves,
// 32 KB), which also stages dQ for the reduce-add in two rounds of 64 columns.
//
// Per query tile t the MMA thread issues: [even t > 0: S^T_t, after the pair's
// dQ was read out] dP^T_t, then (P^T_t and dS^T_t written) dV_c += P^T_t
// dO_t[:, c], [even t: S^T_{t+1} into the columns dV has just read], dK_c +=
// dS^T_t Q_t[:, c], [odd t or the last tile: dQ of the pair].
//
// Warp roles (192 threads): warps 0-3 elementwise (one thread per key row =
// TMEM lane; for dQ, one per query row of the pair), warp 4 TMEM owner and
// MMA issuer, warp 5 TMA.  Every mbarrier wait is bounded and each barrier is
// waited phase by phase.
#pragma once

#include "fa2_bwd.cuh"

namespace fa2 {

struct Bwd256Config {
  static constexpr int D = 256;
  static constexpr int DH = 128;     // output columns per CTA (one half of d)
  static constexpr int T = 128;      // keys per CTA (M of S^T, dP^T, dV, dK)
  static constexpr int TQ = 64;      // query rows per tile (N of S^T, dP^T)
  static constexpr int THREADS = 192;
  static constexpr int MMA_WARP = 4;
  static constexpr int TMA_WARP = 5;
  static constexpr int QSTAGES = 2;
  static constexpr int DOSTAGES = 2;
  static constexpr uint32_t K_BYTES = T * D * 2;         // 64 KB: four 64-column blocks of 128 rows
  static constexpr uint32_t QT_BYTES = TQ * D * 2;       // 32 KB: four 64-column blocks of 64 rows
  static constexpr uint32_t KBLK = T * 128;              // one 64-column block of K_j
  static constexpr uint32_t QBLK = TQ * 128;             // one 64-column block of Q_t / dO_t
  static constexpr uint32_t DS_HALF = T * 128;           // 128 key rows x 64 queries, 16-bit
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_Q = OFF_K + K_BYTES;                // + stage * QT_BYTES
  static constexpr uint32_t OFF_DO = OFF_Q + QSTAGES * QT_BYTES;    // + stage * QT_BYTES
  static constexpr uint32_t OFF_DS = OFF_DO + DOSTAGES * QT_BYTES;  // two halves (tile parity)
  static constexpr uint32_t OFF_BAR = OFF_DS + 2 * DS_HALF;
  static constexpr uint32_t NUM_BARS = 19;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 64 + 4 * kPackedScanWords + 1024;   // misc, scan
  static constexpr uint32_t TMEM_DV = 0;
  static constexpr uint32_t TMEM_DK = 128;
  static constexpr uint32_t TMEM_S = 256;    // S^T, then P^T in its first 32 columns; the pair's dQ from here
  static constexpr uint32_t TMEM_DP = 320;   // dP^T, then dS^T
  static constexpr uint32_t TMEM_V = 384;    // V_j, 16-bit pairs
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

enum : int { BB_V = 18 };   // V_j written to tensor memory (four warp arrivals)

// K_j and Q_t / dO_t tiles: d = 256 as four 64-column boxes each.
template <class C>
__device__ __forceinline__ void bwd256_producer(const BwdCtx& t, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                                const CUtensorMap* tm_do, bool first) {
  const int h = t.seq.h, b = t.seq.b;
  auto load_q = [&](int it) {
    const int s = it % C::QSTAGES;
    mbar_arrive_expect_tx(t.bar(BB_Q + s), C::QT_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sQ + s * C::QT_BYTES + kb * C::QBLK, tm_q, t.merged, kb * 64,
                    t.seq.row0_q + (t.i0 + it) * C::TQ, h, b, t.hb, t.bar(BB_Q + s));
  };
  auto load_do = [&](int it) {
    const int s = it % C::DOSTAGES;
    mbar_arrive_expect_tx(t.bar(BB_DO + s), C::QT_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sDO + s * C::QT_BYTES + kb * C::QBLK, tm_do, t.merged, kb * 64,
                    t.seq.row0_q + (t.i0 + it) * C::TQ, h, b, t.hb, t.bar(BB_DO + s));
  };
  // first pass (before the set-up barrier): K_j and tile 0's Q and dO
  if (first) {
    mbar_arrive_expect_tx(t.bar(BB_KV), C::K_BYTES);
    for (int kb = 0; kb < C::D / 64; ++kb)
      tma_load_rows(t.sK + kb * C::KBLK, tm_k, t.merged, kb * 64, t.seq.row0_k + t.j0, h, b, t.hb, t.bar(BB_KV));
    load_q(0);
    load_do(0);
    return;
  }
  int loaded_q = 1, loaded_do = 1;
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
__device__ __forceinline__ void bwd256_mma(const BwdCtx& t, int dhalf) {
  constexpr uint32_t idesc_s = make_idesc_f16(128, C::TQ, BF16, false, false);    // S^T, dP^T (N = 64 queries)
  constexpr uint32_t idesc_acc = make_idesc_f16(128, C::DH, BF16, false, true);   // dV, dK: A in TMEM, B MN-major
  constexpr uint32_t idesc_dq = make_idesc_f16(128, C::DH, BF16, true, true);     // dQ: A, B MN-major
  const uint64_t k_kmaj = make_sdesc_sw128(t.sK, 16, 1024);
  const uint64_t q_kmaj0 = make_sdesc_sw128(t.sQ, 16, 1024);
  const uint64_t do_kmaj0 = make_sdesc_sw128(t.sDO, 16, 1024);
  // half c of Q_t / dO_t / K_j: its two 64-column blocks, N-adjacent at the block stride
  const uint64_t q_mn0 = make_sdesc_sw128(t.sQ + 2 * dhalf * C::QBLK, C::QBLK, 1024);
  const uint64_t do_mn0 = make_sdesc_sw128(t.sDO + 2 * dhalf * C::QBLK, C::QBLK, 1024);
  const uint64_t k_mn = make_sdesc_sw128(t.sK + 2 * dhalf * C::KBLK, C::KBLK, 1024);
  const uint64_t ds_mn = make_sdesc_sw128(t.sDS, C::DS_HALF, 1024);   // the pair's 128 queries: 2 halves
  const uint32_t tS = t.tmem + C::TMEM_S, tDP = t.tmem + C::TMEM_DP, tV = t.tmem + C::TMEM_V;
  const uint32_t tDV = t.tmem + C::TMEM_DV, tDK = t.tmem + C::TMEM_DK;
  auto issue_s = [&](int it) -> bool {   // S^T = K_j Q_t^T (K = d = 256: 16 steps)
    const int qs = it % C::QSTAGES;
    if (!wait_or_abort(t.bar(BB_Q + qs), (uint32_t)(it / C::QSTAGES) & 1, t.abort_flag, t.status, kSiteMmaQ))
      return false;
    tc_fence_after();
    const uint64_t q_kmaj = q_kmaj0 + (uint64_t)((qs * C::QT_BYTES) >> 4);
#pragma unroll
    for (int k = 0; k < C::D / 16; ++k)
      umma_ss(tS, k_kmaj + kmajor_step<C>(k, C::T), q_kmaj + kmajor_step<C>(k, C::TQ), idesc_s, k > 0 ? 1u : 0u);
    umma_commit(t.bar(BB_S));
    return true;
  };
  bool ok = wait_or_abort(t.bar(BB_KV), 0, t.abort_flag, t.status, kSiteMmaK) &&
            wait_or_abort(t.bar(BB_V), 0, t.abort_flag, t.status, kSiteMmaV);
  if (ok) {
    tc_fence_after();
    ok = issue_s(0);
  }
  for (int it = 0; it < t.niter && ok; ++it) {
    const uint32_t ph = (uint32_t)it & 1;
    const int qs = it % C::QSTAGES, ds = it % C::DOSTAGES;
    const uint64_t do_kmaj = do_kmaj0 + (uint64_t)((ds * C::QT_BYTES) >> 4);
    const uint64_t q_mn = q_mn0 + (uint64_t)((qs * C::QT_BYTES) >> 4);
    const uint64_t do_mn = do_mn0 + (uint64_t)((ds * C::QT_BYTES) >> 4);
    // an even tile after the first: the previous pair's dQ occupies the S^T and
    // dP^T columns until the elementwise warps have read it out
    if ((it & 1) == 0 && it > 0) {
      if (!wait_or_abort(t.bar(BB_DQEMPTY), (uint32_t)((it >> 1) - 1) & 1, t.abort_flag, t.status, kSiteMmaO)) break;
      tc_fence_after();
      if (!issue_s(it)) break;
    }
    if (!wait_or_abort(t.bar(BB_DO + ds), (uint32_t)(it / C::DOSTAGES) & 1, t.abort_flag, t.status, kSiteMmaQ)) break;
    tc_fence_after();
    // dP^T = V_j dO_t^T: A = V_j from tensor memory, 8 columns per K step of 16
#pragma unroll
    for (int k = 0; k < C::D / 16; ++k)
      umma_ts(tDP, tV + (uint32_t)(k * 8), do_kmaj + kmajor_step<C>(k, C::TQ), idesc_s, k > 0 ? 1u : 0u);
    umma_commit(t.bar(BB_DP));
    if (!wait_or_abort(t.bar(BB_P), ph, t.abort_flag, t.status, kSiteMmaP)) break;
    tc_fence_after();
    // K = 64 queries in steps of 16: P^T / dS^T sit in the first 32 columns
#pragma unroll
    for (int k = 0; k < C::TQ / 16; ++k)
      umma_ts(tDV, tS + (uint32_t)(k * 8), do_mn + (uint64_t)((k * 16 * 128) >> 4), idesc_acc,
              (it > 0 || k > 0) ? 1u : 0u);
    umma_commit(t.bar(BB_DOEMPTY + ds));
    // S^T of the next tile (odd) overwrites the P^T columns dV has just read
    // (the MMAs of one thread execute in order)
    if ((it & 1) == 0 && it + 1 < t.niter && !issue_s(it + 1)) break;
#pragma unroll
    for (int k = 0; k < C::TQ / 16; ++k)
      umma_ts(tDK, tDP + (uint32_t)(k * 8), q_mn + (uint64_t)((k * 16 * 128) >> 4), idesc_acc,
              (it > 0 || k > 0) ? 1u : 0u);
    umma_commit(t.bar(BB_QEMPTY + qs));
    // dQ of the pair (2p, 2p + 1) = dS K_j[:, c], M = 128 queries, N = 128, into
    // the S^T and dP^T columns (dV and dK above read P^T and dS^T first; S^T of
    // the next tile waits for the read-out)
    if ((it & 1) == 1 || it + 1 == t.niter) {
#pragma unroll
      for (int k = 0; k < C::T / 16; ++k)
        umma_ss(tS, ds_mn + (uint64_t)((k * 16 * 128) >> 4), k_mn + (uint64_t)((k * 16 * 128) >> 4), idesc_dq,
                k > 0 ? 1u : 0u);
      umma_commit(t.bar(BB_DQ));
    }
  }
  if (ok) umma_commit(t.bar(BB_END));
  umma_commit(t.bar(BB_EXIT));
  wait_drain(t.bar(BB_EXIT), 0, t.status);
}

template <class C, bool BF16>
__device__ __forceinline__ void bwd256_elementwise(const BwdCtx& t, const BwdParams& p, const KeyMask& km,
                                                   uint8_t* smem, int warp, int lane, int dhalf,
                                                   const CUtensorMap* tm_dq) {
  const KernelParams& f = p.f;
  const int quad = warp & 3;
  const int r = quad * 32 + lane;          // TMEM lane: key row (S^T, dP^T, dK, dV, V) or query row of the pair (dQ)
  const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
  const uint32_t tS = t.tmem + lane_off + C::TMEM_S;
  const uint32_t tDP = t.tmem + lane_off + C::TMEM_DP;
  const int n_q = t.seq.n_q;
  const int key = t.j0 + r;
  // V_j row `key` into tensor memory as 16-bit pairs (zeros past the sequence)
  {
    const uint4* src = reinterpret_cast<const uint4*>(
        reinterpret_cast<const uint8_t*>(p.v) +
        2 * ((long long)t.seq.b * p.v_bs + (long long)t.seq.h * p.v_hs + (long long)(t.seq.row0_k + key) * p.v_rs));
    const bool live = key < t.seq.n_k;
#pragma unroll 1
    for (int c = 0; c < C::D / 2; c += 32) {   // 32 columns = 64 elements = 8 uint4 per round
      uint32_t w[32];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint4 x = live ? __ldg(src + c / 4 + i) : make_uint4(0u, 0u, 0u, 0u);
        w[4 * i] = x.x;
        w[4 * i + 1] = x.y;
        w[4 * i + 2] = x.z;
        w[4 * i + 3] = x.w;
      }
      tmem_st_32x32b_x32(t.tmem + lane_off + C::TMEM_V + c, w);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(t.bar(BB_V));
  }
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
  // dQ of pair pr (query tiles 2pr, 2pr + 1 from i0), columns [128 c, 128 c +
  // 128): read out of TMEM in two rounds of 64 columns, staged in this warp's
  // own rows of the two dS^T halves (box b = columns [32 b, 32 b + 32) of the
  // round in half b) and added to the fp32 accumulator by TMA.  A lone last
  // tile's pair keeps rows 0-63 only.  The columns are freed after the second
  // round's load.
  auto dq_out = [&](int pr, bool lone) -> bool {
    bool w = wait_or_abort(t.bar(BB_DQ), (uint32_t)pr & 1, t.abort_flag, t.status, kSiteEpilogueO);
    w = __all_sync(0xffffffffu, w);
    if (!w) return false;
    tc_fence_after();
    const int y = t.seq.row0_q + (t.i0 + 2 * pr) * C::TQ + quad * 32;   // rows past the tensor are clipped
#pragma unroll 1
    for (int round = 0; round < 2; ++round) {
      uint32_t dq[64];
      tmem_ld_32x32b_x32(tS + 64 * round, dq);
      tmem_ld_32x32b_x32(tS + 64 * round + 32, dq + 32);
      tmem_ld_wait_x32(dq);
      tmem_ld_wait_x32(dq + 32);
      if (round == 1) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(t.bar(BB_DQEMPTY));
      }
      // this warp's boxes of the previous round (or pair) were read out
      if (lane == 0) bulk_wait_read_all();
      __syncwarp();
      if (lone && quad >= 2) continue;    // rows of the pair's missing second tile
#pragma unroll
      for (int b = 0; b < 2; ++b) {
        uint8_t* row = smem + C::OFF_DS + b * C::DS_HALF + quad * 4096 + lane * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(row + ((c ^ (lane & 7)) * 16)) =
              make_uint4(dq[32 * b + 4 * c], dq[32 * b + 4 * c + 1], dq[32 * b + 4 * c + 2], dq[32 * b + 4 * c + 3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int b = 0; b < 2; ++b)
          tma_reduce_add_3d(tm_dq, smem_u32(smem + C::OFF_DS + b * C::DS_HALF + quad * 4096),
                            C::DH * dhalf + 64 * round + 32 * b, y, t.hb);
        bulk_commit_group();
      }
    }
    return true;
  };
  bool ok = true;
  for (int it = 0; it < t.niter; ++it) {
    const uint32_t ph = (uint32_t)it & 1;
    const int q0 = (t.i0 + it) * C::TQ;   // first query of the tile
    // the previous pair's dQ: its columns hold this tile's S^T once read out
    if ((it & 1) == 0 && it > 0 && !dq_out((it >> 1) - 1, false)) {
      ok = false;
      break;
    }
    // L (exp2 domain) and D of the 64 queries: lane c holds queries c and
    // c + 32, every lane takes each value by shuffle
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
    // hidden pairs (and rows without keys) give 0, in a pass of its own that
    // only blocks some pair of which is hidden run
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
    // dS^T row to the tile's half of the shared buffer (128-byte swizzle),
    // once TMA has read out this warp's dQ boxes of the previous pair (they
    // sit in this warp's rows of both halves)
    if (lane == 0) bulk_wait_read_all();
    __syncwarp();
    uint8_t* ds_row = smem + C::OFF_DS + (it & 1) * C::DS_HALF + r * 128;
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
  }
  if (ok && t.niter > 0) ok = dq_out((t.niter - 1) >> 1, (t.niter & 1) == 1);
  if (lane == 0) bulk_wait_all();   // this warp's reduce-adds performed before the CTA exits
  __syncwarp();
  if (ok && t.niter > 0) {
    ok = wait_or_abort(t.bar(BB_END), 0, t.abort_flag, t.status, kSiteDrain);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) return;
  tc_fence_after();
  // dV_j and dK_j rows (lane = key row), columns [128 c, 128 c + 128); zero
  // when no query row sees the tile
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const uint32_t base = t.tmem + lane_off + (which ? C::TMEM_DK : C::TMEM_DV);
    uint8_t* out = reinterpret_cast<uint8_t*>(which ? p.dk : p.dv) +
                   2 * ((which ? (long long)t.seq.b * p.k_bs + (long long)t.seq.h * p.k_hs +
                                     (long long)(t.seq.row0_k + key) * p.k_rs
                               : (long long)t.seq.b * p.v_bs + (long long)t.seq.h * p.v_hs +
                                     (long long)(t.seq.row0_k + key) * p.v_rs) +
                        (long long)C::DH * dhalf);
#pragma unroll 1
    for (int c = 0; c < C::DH; c += 32) {
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

// One CTA per (key tile, half dhalf of d); blocks 2u and 2u + 1 are the two halves
// of the key tile the forward kernels' unit order gives block u.  PACKED: a
// packed batch whose grid holds only its real key tiles, as in fa2_bwd_kernel.
template <bool BF16, bool PACKED>
__global__ void __launch_bounds__(192, 1)
    fa2_bwd256_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_dq,
                      const BwdParams p) {
  using C = Bwd256Config;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);
  const KernelParams& f = p.f;
  const int dhalf = (int)(blockIdx.x & 1u);
  const int block = (int)(blockIdx.x >> 1);

  BwdCtx t;
  int bh, unit;
  int units = p.num_k_tiles;
  if constexpr (PACKED) {
    if (!packed_unit<C::THREADS>(f, C::T, true, p.num_k_tiles, 4, reinterpret_cast<int*>(smem + C::OFF_MISC + 64),
                                 t.seq, unit, units, block))
      return;
  } else {
    unit_of_block(block, f.bh, p.num_k_tiles, bh, unit, 4);
    if (!seq_info(f, bh, t.seq)) return;
    if (t.seq.n_k > p.num_k_tiles * C::T) {
      if (threadIdx.x == 0 && unit == 0 && dhalf == 0) atomicOr(f.status, kStatusBadSeqlens);
      return;
    }
  }
  const int jt = units - 1 - unit;   // the key tiles with the most query tiles start first
  t.j0 = jt * C::T;
  if (t.j0 >= t.seq.n_k) return;
  const KeyMask km = key_mask(f, t.seq);
  {
    int r_lo, r_hi;
    queries_of_tile(km, t.seq.n_q, t.j0, min(t.j0 + C::T, t.seq.n_k) - 1, r_lo, r_hi);
    t.i0 = r_lo <= r_hi ? r_lo / C::TQ : 0;
    t.niter = r_lo <= r_hi ? r_hi / C::TQ - t.i0 + 1 : 0;
  }
  t.hb = t.seq.b * f.heads + t.seq.h;
  t.merged = f.merged_bh != 0;
  t.bar0 = sbase + C::OFF_BAR;
  t.sK = sbase + C::OFF_K;
  t.sV = 0;   // V_j lives in tensor memory
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
    mbar_init(t.bar(BB_P), 4);         // one arrival per elementwise warp
    mbar_init(t.bar(BB_DQ), 1);
    mbar_init(t.bar(BB_DQEMPTY), 4);
    mbar_init(t.bar(BB_END), 1);
    mbar_init(t.bar(BB_EXIT), 1);
    mbar_init(t.bar(BB_V), 4);
    *abort_flag = 0;
    fence_mbar_init();
    fence_proxy_async_smem();   // the initialised barriers, before this thread's own TMA loads signal them
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_dq);
    if (t.niter > 0) bwd256_producer<C>(t, &tm_q, &tm_k, &tm_do, true);
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
    if (lane == 0 && t.niter > 0) bwd256_producer<C>(t, &tm_q, &tm_k, &tm_do, false);
  } else if (warp == C::MMA_WARP) {
    if (lane == 0 && t.niter > 0) bwd256_mma<C, BF16>(t, dhalf);
    __syncwarp();
  } else {
    bwd256_elementwise<C, BF16>(t, p, km, smem, warp, lane, dhalf, &tm_dq);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(t.tmem, C::TMEM_COLS);
  }
}

template <bool BF16, bool PACKED>
int launch_bwd256_main(const BwdLaunchArgs& a) {
  using C = Bwd256Config;
  auto kern = fa2_bwd256_kernel<BF16, PACKED>;
  static std::atomic<unsigned long long> configured{0};
  const int e = once_per_device(configured, [&]() -> int {
    return (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  });
  if (e != 0) return e;
  const long long blocks =
      2 * (PACKED ? (long long)a.p.f.heads * a.p.f.packed_units : (long long)a.p.f.bh * a.p.num_k_tiles);
  kern<<<(unsigned)blocks, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tm_q, a.tm_k, a.tm_do, a.tm_dq, a.p);
  return (int)cudaGetLastError();
}

// D / accumulator zeroing, the main kernel, then the 16-bit dQ conversion;
// maps: q and dout boxes of 64 rows, k of 128 rows, dQ 32 x 32 fp32.
template <bool BF16>
int launch_bwd256_dtype(const BwdLaunchArgs& a) {
  using C = Bwd256Config;
  const long long rows = a.p.slices * a.p.f.total_q;
  {
    const long long threads = rows * (C::D / 8);
    fa2_bwd_preprocess_kernel<256, BF16><<<(unsigned)((threads + 255) / 256), 256, 0, a.stream>>>(a.p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return (int)e;
  }
  const int e = a.p.f.packed_units ? launch_bwd256_main<BF16, true>(a) : launch_bwd256_main<BF16, false>(a);
  if (e != 0) return e;
  const long long n8 = rows * (C::D / 8);
  fa2_bwd_dq_convert_kernel<256, BF16><<<(unsigned)((n8 + 255) / 256), 256, 0, a.stream>>>(a.p);
  return (int)cudaGetLastError();
}

}  // namespace fa2
