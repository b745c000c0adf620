// fa2_decode.cuh -- forward pass for a few query rows against many keys (the
// decoding regime: one new token, or a handful, attending to a long cache).
//
// With N_q <= 8 rows per sequence there is no query tile to fill a tensor
// core, and the step is bound by reading K and V from HBM once: each key
// costs 4 d bytes (16-bit K and V) against 4 d FLOPs per query row.  So the
// keys of each (batch, head) are split into chunks, one CTA per chunk,
// enough CTAs to cover every SM twice, and each chunk is reduced on CUDA
// cores to the online-softmax state of every query row -- local maximum m,
// l = sum 2^(s - m), O~ = sum 2^(s - m) v -- which a second kernel merges
// with the same rescaling step the tiled loop applies between key tiles:
// M = max m_c, l = sum 2^(m_c - M) l_c, O = sum 2^(m_c - M) O~_c / l (Lesson
// 6.6, "Online softmax"; FlashAttention V2 in depth, section 3.2).  Lesson
// 6.6 ("Common misconceptions") names this regime as needing its own kernel.
// This CUDA-core kernel serves one query row at d = 64 and every row count at
// d = 256; otherwise the tiled tensor-core kernel reduces the chunks
// (fa2_decode_tc.cuh), since the per-key products grow with the rows.
//
// Per CTA: a TMA warp streams [BLOCK x d] boxes of K and V through a 3-stage
// shared-memory ring; four compute warps each take BLOCK/4 keys of a stage.
// A key row is spread over d/8 lanes (16 bytes each), so a lane keeps only
// its 8 elements of each query row in registers; the partial dot products
// of all rows are summed across those lanes by a reduce-scatter that leaves
// each lane the score of one row, whose online-softmax state that lane keeps
// (one exponential per lane per key); p then goes back to every lane for
// its part of O~.  The running maximum is raised only past a 2^8 margin (as
// in the tiled kernels), so rescaling O~ is rare.  At the end the per-lane-group states are merged through the
// (then idle) stage buffers and written to the caller's workspace.
#pragma once

#include "fa2_common.cuh"

namespace fa2 {

struct DecodeParams {
  const void* q;                 // query rows, 16-bit
  long long q_bs, q_hs, q_rs;    // q strides in elements (head-dim stride 1)
  float* ws_o;                   // [B*H][n_q][splits][d] partial O~
  float* ws_ml;                  // [B*H][n_q][splits][2] partial (m, l), exp2 domain
  int splits;                    // key chunks per (b, h)
  int chunk;                     // keys per chunk (a multiple of the stage size)
  int base;                      // first key of chunk 0: keys before it are seen by no row
  KernelParams f;                // outputs, offsets, sizes, mask, scale (as the tiled kernels)
};

struct DecodeLaunchArgs {
  CUtensorMap tm_k, tm_v;        // boxes of d columns x BLOCK rows, no swizzle
  DecodeParams p;
  bool bf16;
  cudaStream_t stream;
};

constexpr int kDecodeMaxRows = 8;  // FA2_DECODE_MAX_Q
constexpr float kRescaleDecodeLog2 = 8.0f;   // raise the running maximum only past a 2^8 margin

template <int D_>
struct DecodeConfig {
  static constexpr int D = D_;
  static constexpr int G = D / 8;                      // lanes per key row (16 bytes each)
  static constexpr int KPW = 32 / G;                   // keys a warp takes per step
  static constexpr int WARPS = 4;                      // compute warps
  static constexpr int TMA_WARP = WARPS;
  static constexpr int THREADS = (WARPS + 1) * 32;
  static constexpr int BLOCK = decode_block_rows(D);   // keys per stage
  static constexpr int KEYS_PER_WARP = BLOCK / WARPS;
  static constexpr int STEPS = KEYS_PER_WARP / KPW;    // steps per warp per stage
  static constexpr int STAGES = 3;
  static constexpr int GROUPS = WARPS * KPW;           // lane groups in the CTA, each with its own state
  static constexpr uint32_t TILE_BYTES = BLOCK * D * 2;
  static constexpr uint32_t OFF_K = 0;
  static constexpr uint32_t OFF_V = STAGES * TILE_BYTES;
  static constexpr uint32_t OFF_BAR = 2 * STAGES * TILE_BYTES;
  static constexpr uint32_t NUM_BARS = 2 * STAGES + 2;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 128;   // + alignment slack
  // merge area (reuses the stage buffers once every stage is consumed)
  static constexpr uint32_t MERGE_O_BYTES = GROUPS * kDecodeMaxRows * D * 4;
  static constexpr uint32_t MERGE_ML_BYTES = GROUPS * kDecodeMaxRows * 2 * 4;
  static_assert(KEYS_PER_WARP % KPW == 0, "keys per warp");
  static_assert(MERGE_O_BYTES + MERGE_ML_BYTES <= 2 * STAGES * TILE_BYTES, "merge area");
  static_assert(2 * SMEM_BYTES <= 232448, "two CTAs per SM");
};

enum : int {
  DC_FULL = 0,                   // + stage: K and V of the stage landed
  DC_EMPTY = 3,                  // + stage: four compute warps are done with it
  DC_DONE = 6,                   // every compute warp has finished reading stages
  DC_MERGED = 7,                 // every lane group's state is in the merge area
};

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4& u, float* x) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = unpack2<BF16>(w[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

// The chunk of keys [c0, c1) one CTA reduces, within a sequence, clipped to
// the keys some query row sees; false if empty.
__device__ __forceinline__ bool decode_range(const KeyMask& km, int n_q, int split, int chunk, int base, int& c0,
                                             int& c1) {
  int lo, end;
  if (!km.tile_range<true>(0, n_q - 1, lo, end)) return false;
  c0 = max(lo, base + split * chunk);
  c1 = min(end, min(km.n_k, base + (split + 1) * chunk));
  return c1 > c0;
}

// Lane (within its group of G) that owns query row r after dc_reduce_scatter.
template <int NQ, int G>
__device__ __forceinline__ constexpr int dc_owner(int r) {
  int li = 0;
  for (int rd = 0, w = NQ; w > 1; ++rd, w >>= 1)
    if ((r / (w / 2)) & 1) li += G >> (rd + 1);   // which half of the current rows r lies in
  return li;
}

// Sum partial dot products over the G lanes of a group so that each lane ends
// with the full sum for one row (lanes own rows in halving steps: a lane keeps
// one half of the rows and passes the other half to its partner, then the
// last lanes sharing a row add up): log2(G) shuffles instead of NQ log2(G).
// Returns the lane's row; v[0] holds its sum.
template <int NQ, int G>
__device__ __forceinline__ int dc_reduce_scatter(float* v, int li) {
  int own = 0;
#pragma unroll
  for (int rd = 0, w = NQ; w > 1; ++rd, w >>= 1) {
    const int mask = G >> (rd + 1);
    const bool upper = (li & mask) != 0;
    const int half = w / 2;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = upper ? v[i] : v[i + half];
      const float keep = upper ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, mask);
    }
    if (upper) own += half;
  }
#pragma unroll
  for (int mask = G / NQ / 2; mask >= 1; mask >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], mask);
  return own;
}

template <int NQ, class C, bool BF16>
__device__ __forceinline__ void dc_compute(const DecodeParams& dp, const SeqInfo& seq, const KeyMask& km, int n_q,
                                           int c0, int c1, uint32_t sbase, uint32_t bar0, volatile int* abort_flag,
                                           int warp, int lane, float* st_m, float* st_l, float* st_o) {
  static_assert(NQ <= C::G, "one row per lane after the reduce-scatter");
  const KernelParams& p = dp.f;
  const int g = lane / C::G;            // lane group within the warp (its key of a step)
  const int li = lane % C::G;           // lane within the group
  const int gbase = g * C::G;
  const int e0 = li * 8;                // this lane's 8 elements of a row
  // this lane's slice of every query row (exp2 domain), as fp32 pairs
  float2 q[NQ][4];
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    float x[8];
    if (r < n_q) {
      const uint8_t* src = reinterpret_cast<const uint8_t*>(dp.q) +
                           2 * ((long long)seq.b * dp.q_bs + (long long)seq.h * dp.q_hs +
                                (long long)(seq.row0_q + r) * dp.q_rs + e0);
      unpack8<BF16>(*reinterpret_cast<const uint4*>(src), x);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] = 0.f;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) q[r][e] = make_float2(x[2 * e] * p.scale_log2, x[2 * e + 1] * p.scale_log2);
  }
  // the row this lane owns after the reduce-scatter, and that row's band;
  // rows past n_q repeat the last row's band (computed, never stored)
  int own = 0;   // as dc_reduce_scatter assigns it (it depends on the lane only)
#pragma unroll
  for (int rd = 0, w = NQ; w > 1; ++rd, w >>= 1)
    if (li & (C::G >> (rd + 1))) own += w / 2;
  const int own_row = min(own, n_q - 1);
  const int own_lo = km.row_lo(own_row), own_hi = km.row_hi(own_row);
  // a stage needs no per-key mask when it ends before c1 and every row sees all of it
  const int lo_last = km.row_lo(n_q - 1);
  const int hi_first = km.row_hi(0);
  float m = -INFINITY, l = 0.f;   // the owned row's state (exp2 domain)
  float2 o[NQ][4];                 // every row's 8 output elements of this lane
#pragma unroll
  for (int r = 0; r < NQ; ++r)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[r][e] = make_float2(0.f, 0.f);
  const int nblk = (c1 - c0 + C::BLOCK - 1) / C::BLOCK;
  bool ok = true;
  for (int b = 0; b < nblk; ++b) {
    const int s = b % C::STAGES;
    ok = wait_or_abort(bar0 + 8u * (DC_FULL + s), (uint32_t)(b / C::STAGES) & 1, abort_flag, p.status,
                       kSiteDecodeFull);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    const int kb0 = c0 + b * C::BLOCK;
    const int kb1 = kb0 + C::BLOCK;
    const bool full = kb1 <= c1 && (kb1 <= km.pre_end || (kb0 >= lo_last && kb1 - 1 <= hi_first));
    const uint32_t sK = sbase + C::OFF_K + s * C::TILE_BYTES;
    const uint32_t sV = sbase + C::OFF_V + s * C::TILE_BYTES;
#pragma unroll 2
    for (int step = 0; step < C::STEPS; ++step) {
      const int kl = warp * C::KEYS_PER_WARP + step * C::KPW + g;   // key within the stage
      const int key = kb0 + kl;
      const uint4 kr = lds128(sK + kl * (C::D * 2) + e0 * 2);
      const float2 k0 = unpack2<BF16>(kr.x), k1 = unpack2<BF16>(kr.y), k2 = unpack2<BF16>(kr.z),
                   k3 = unpack2<BF16>(kr.w);
      float v[NQ];
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        float2 a = __fmul2_rn(q[r][0], k0);
        a = __ffma2_rn(q[r][1], k1, a);
        a = __ffma2_rn(q[r][2], k2, a);
        a = __ffma2_rn(q[r][3], k3, a);
        v[r] = a.x + a.y;
      }
      dc_reduce_scatter<NQ, C::G>(v, li);
      float sc = v[0];   // the owned row's score for this key
      if (!full) {
        const bool vis = key < c1 && (key < km.pre_end || (key >= own_lo && key <= own_hi));
        if (!vis) sc = -INFINITY;
      }
      // raise the maximum past a 2^8 margin (rare after the first key): every
      // lane then rescales its elements of the rows whose owners raised (with
      // one row every lane holds that row's state and rescales on its own)
      const bool raise = sc > m + kRescaleDecodeLog2;
      if (NQ == 1) {
        if (raise) {
          const float alpha = ex2_approx(m - sc);   // 0 when m was -inf
          m = sc;
          l *= alpha;
          const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
          for (int e = 0; e < 4; ++e) o[0][e] = __fmul2_rn(o[0][e], a2);
        }
      } else if (__any_sync(0xffffffffu, raise)) {
        const float alpha = raise ? ex2_approx(m - sc) : 1.f;   // 0 when m was -inf
        if (raise) {
          m = sc;
          l *= alpha;
        }
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
          const float ar = __shfl_sync(0xffffffffu, alpha, gbase + dc_owner<NQ, C::G>(r));
          const float2 a2 = make_float2(ar, ar);
#pragma unroll
          for (int e = 0; e < 4; ++e) o[r][e] = __fmul2_rn(o[r][e], a2);
        }
      }
      const float pown = ex2_approx(sc - (m == -INFINITY ? 0.f : m));   // 0 for a hidden key
      l += pown;
      const uint4 vr = lds128(sV + kl * (C::D * 2) + e0 * 2);
      const float2 v0 = unpack2<BF16>(vr.x), v1 = unpack2<BF16>(vr.y), v2 = unpack2<BF16>(vr.z),
                   v3 = unpack2<BF16>(vr.w);
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float pr = NQ == 1 ? pown : __shfl_sync(0xffffffffu, pown, gbase + dc_owner<NQ, C::G>(r));
        const float2 p2 = make_float2(pr, pr);
        o[r][0] = __ffma2_rn(p2, v0, o[r][0]);
        o[r][1] = __ffma2_rn(p2, v1, o[r][1]);
        o[r][2] = __ffma2_rn(p2, v2, o[r][2]);
        o[r][3] = __ffma2_rn(p2, v3, o[r][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar0 + 8u * (DC_EMPTY + s));
  }
  // every stage consumed: the stage buffers become the merge area
  if (lane == 0) mbar_arrive(bar0 + 8u * DC_DONE);
  if (ok) ok = wait_or_abort(bar0 + 8u * DC_DONE, 0, abort_flag, p.status, kSiteDecodeMerge);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) return;
  const int grp = warp * C::KPW + g;
  if (li == dc_owner<NQ, C::G>(own)) {   // one lane per owned row writes its state
    st_m[grp * kDecodeMaxRows + own] = m;
    st_l[grp * kDecodeMaxRows + own] = l;
  }
#pragma unroll
  for (int r = 0; r < NQ; ++r) {
    float4* dst = reinterpret_cast<float4*>(st_o + ((size_t)grp * kDecodeMaxRows + r) * C::D + e0);
    dst[0] = make_float4(o[r][0].x, o[r][0].y, o[r][1].x, o[r][1].y);
    dst[1] = make_float4(o[r][2].x, o[r][2].y, o[r][3].x, o[r][3].y);
  }
}

// Merge the CTA's lane-group states and write its partial for every query row.
template <class C>
__device__ __forceinline__ void dc_write_partial(const DecodeParams& dp, int bh, int split, int n_q, const float* st_m,
                                                 const float* st_l, const float* st_o, bool empty, int tid) {
  for (int idx = tid; idx < n_q * C::D; idx += C::WARPS * 32) {
    const int r = idx / C::D, c = idx - r * C::D;
    float M = -INFINITY, L = 0.f, O = 0.f;
    if (!empty) {
#pragma unroll
      for (int gi = 0; gi < C::GROUPS; ++gi) M = fmaxf(M, st_m[gi * kDecodeMaxRows + r]);
      if (M != -INFINITY) {
#pragma unroll
        for (int gi = 0; gi < C::GROUPS; ++gi) {
          const float mg = st_m[gi * kDecodeMaxRows + r];
          const float f = mg == -INFINITY ? 0.f : ex2_approx(mg - M);
          L = fmaf(f, st_l[gi * kDecodeMaxRows + r], L);
          O = fmaf(f, st_o[((size_t)gi * kDecodeMaxRows + r) * C::D + c], O);
        }
      }
    }
    const size_t slot = ((size_t)bh * dp.f.n_q + r) * dp.splits + split;
    dp.ws_o[slot * C::D + c] = O;
    if (c == 0) {
      dp.ws_ml[slot * 2] = M;
      dp.ws_ml[slot * 2 + 1] = L;
    }
  }
}

// Two CTAs per SM for every row count: with eight rows (8 x 8 elements of q
// and O~ per lane) that costs a few spilled registers but hides twice the
// latency, which measured faster than one CTA per SM with none.
template <int D, bool BF16, int NQ>
__global__ void __launch_bounds__(DecodeConfig<D>::THREADS, 2)
    fa2_decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const DecodeParams dp) {
  using C = DecodeConfig<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((128u - (raw_addr & 127u)) & 127u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC);
  const int warp = (int)(threadIdx.x >> 5);
  const int lane = (int)(threadIdx.x & 31);
  const KernelParams& p = dp.f;
  grid_launch_dependents();   // the merge kernel may be scheduled now; it waits for this grid's partials

  const int bh = (int)blockIdx.x / dp.splits;
  const int split = (int)blockIdx.x - bh * dp.splits;
  SeqInfo seq;
  if (!seq_info(p, bh, seq)) return;
  if (seq.n_k > dp.base + dp.splits * dp.chunk) {   // a packed sequence longer than the split plan covers
    if (threadIdx.x == 0 && split == 0) atomicOr(p.status, kStatusBadSeqlens);
    return;
  }
  const int n_q = seq.n_q;
  if (n_q == 0) return;
  const KeyMask km = key_mask(p, seq);
  int c0 = 0, c1 = 0;
  const bool empty = !decode_range(km, n_q, split, dp.chunk, dp.base, c0, c1);
  const int nblk = empty ? 0 : (c1 - c0 + C::BLOCK - 1) / C::BLOCK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar0 + 8u * (DC_FULL + s), 1);
      mbar_init(bar0 + 8u * (DC_EMPTY + s), C::WARPS);
    }
    mbar_init(bar0 + 8u * DC_DONE, C::WARPS);
    mbar_init(bar0 + 8u * DC_MERGED, C::WARPS);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == C::TMA_WARP && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  __syncthreads();

  float* st_o = reinterpret_cast<float*>(smem);
  float* st_m = reinterpret_cast<float*>(smem + C::MERGE_O_BYTES);
  float* st_l = st_m + C::GROUPS * kDecodeMaxRows;

  if (warp == C::TMA_WARP) {
    if (lane == 0) {
      const int hb = seq.b * p.heads + seq.h;
      const bool merged = p.merged_bh != 0;
      int last_use[C::STAGES];
      for (int s = 0; s < C::STAGES; ++s) last_use[s] = -1;
      for (int b = 0; b < nblk; ++b) {
        const int s = b % C::STAGES;
        const int w = b / C::STAGES;
        if (w > 0 &&
            !wait_or_abort(bar0 + 8u * (DC_EMPTY + s), (uint32_t)(w - 1) & 1, abort_flag, p.status, kSiteProducerEmpty))
          break;
        const int row = seq.row0_k + c0 + b * C::BLOCK;
        mbar_arrive_expect_tx(bar0 + 8u * (DC_FULL + s), 2 * C::TILE_BYTES);
        tma_load_rows(sbase + C::OFF_K + s * C::TILE_BYTES, &tm_k, merged, 0, row, seq.h, seq.b, hb,
                      bar0 + 8u * (DC_FULL + s));
        tma_load_rows(sbase + C::OFF_V + s * C::TILE_BYTES, &tm_v, merged, 0, row, seq.h, seq.b, hb,
                      bar0 + 8u * (DC_FULL + s));
        last_use[s] = w;
      }
      for (int s = 0; s < C::STAGES; ++s)
        if (last_use[s] >= 0) wait_drain(bar0 + 8u * (DC_FULL + s), (uint32_t)last_use[s] & 1, p.status);
    }
    return;   // the producer takes no part in the merge (no block-wide barrier follows)
  }
  dc_compute<NQ, C, BF16>(dp, seq, km, n_q, c0, c1, sbase, bar0, abort_flag, warp, lane, st_m, st_l, st_o);
  __syncwarp();
  if (lane == 0) mbar_arrive(bar0 + 8u * DC_MERGED);
  bool ok = wait_or_abort(bar0 + 8u * DC_MERGED, 0, abort_flag, p.status, kSiteDecodeMerge);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok || *abort_flag) return;
  dc_write_partial<C>(dp, bh, split, n_q, st_m, st_l, st_o, empty, (int)threadIdx.x);
}

// One block per (b*h, query row): merge the row's partials, store O and LSE.
// Launched right behind the split kernel with programmatic stream
// serialization (launch_decode_merge), so its launch overlaps that kernel's
// last CTAs.
template <int D, bool BF16>
__global__ void __launch_bounds__(128)
    fa2_decode_merge_kernel(const DecodeParams dp) {
  grid_dependency_wait();   // the split kernel's partials are complete and visible
  const KernelParams& p = dp.f;
  const int bh = (int)blockIdx.x / p.n_q;
  const int r = (int)blockIdx.x - bh * p.n_q;
  SeqInfo seq;
  if (!seq_info(p, bh, seq)) return;   // the decode kernel has already reported it
  if (r >= seq.n_q || seq.n_k > dp.base + dp.splits * dp.chunk) return;
  const size_t slot0 = ((size_t)bh * p.n_q + r) * dp.splits;
  float M = -INFINITY;
  for (int s = 0; s < dp.splits; ++s) M = fmaxf(M, dp.ws_ml[(slot0 + s) * 2]);
  float L = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < dp.splits; ++s) {
      const float ms = dp.ws_ml[(slot0 + s) * 2];
      if (ms != -INFINITY) L = fmaf(ex2_approx(ms - M), dp.ws_ml[(slot0 + s) * 2 + 1], L);
    }
  }
  const bool empty = !(L > 0.f);
  const float inv_l = empty ? 0.f : 1.f / L;
  uint8_t* o_row = reinterpret_cast<uint8_t*>(p.o) +
                   2 * ((long long)seq.b * p.o_bs + (long long)seq.h * p.o_hs + (long long)(seq.row0_q + r) * p.o_rs);
  for (int c = 2 * (int)threadIdx.x; c < D; c += 2 * (int)blockDim.x) {
    float a0 = 0.f, a1 = 0.f;
    if (!empty) {
      for (int s = 0; s < dp.splits; ++s) {
        const float ms = dp.ws_ml[(slot0 + s) * 2];
        if (ms == -INFINITY) continue;
        const float f = ex2_approx(ms - M);
        const float2 v = *reinterpret_cast<const float2*>(dp.ws_o + (slot0 + s) * D + c);
        a0 = fmaf(f, v.x, a0);
        a1 = fmaf(f, v.y, a1);
      }
    }
    *reinterpret_cast<uint32_t*>(o_row + 2 * c) = empty ? 0u : pack2<BF16>(a0 * inv_l, a1 * inv_l);
  }
  if (threadIdx.x == 0)
    p.lse[(long long)seq.b * p.l_bs + (long long)seq.h * p.l_hs + seq.row0_q + r] =
        empty ? -INFINITY : (M + log2f(L)) * 0.6931471805599453f;
}

// The merge behind a split kernel on the same stream, as a programmatic
// dependent launch (its blocks wait in grid_dependency_wait for the partials).
template <int D, bool BF16>
int launch_decode_merge(const DecodeParams& dp, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)dp.f.bh * dp.f.n_q));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, fa2_decode_merge_kernel<D, BF16>, dp);
}

template <int D, bool BF16, int NQ>
int launch_decode_nq(const DecodeLaunchArgs& a) {
  using C = DecodeConfig<D>;
  auto kern = fa2_decode_kernel<D, BF16, NQ>;
  static std::atomic<unsigned long long> configured{0};
  const int e = once_per_device(configured, [&]() -> int {
    return (int)cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
  });
  if (e != 0) return e;
  const long long blocks = (long long)a.p.f.bh * a.p.splits;
  kern<<<(unsigned)blocks, C::THREADS, C::SMEM_BYTES, a.stream>>>(a.tm_k, a.tm_v, a.p);
  cudaError_t r = cudaGetLastError();
  if (r != cudaSuccess) return (int)r;
  return launch_decode_merge<D, BF16>(a.p, a.stream);
}

template <int D, bool BF16>
int launch_decode_dtype(const DecodeLaunchArgs& a) {
  const int n = a.p.f.n_q;
  if (n <= 1) return launch_decode_nq<D, BF16, 1>(a);
  if (n <= 2) return launch_decode_nq<D, BF16, 2>(a);
  if (n <= 4) return launch_decode_nq<D, BF16, 4>(a);
  return launch_decode_nq<D, BF16, 8>(a);
}

template <int D>
int launch_decode_dispatch(const DecodeLaunchArgs& a) {
  return a.bf16 ? launch_decode_dtype<D, true>(a) : launch_decode_dtype<D, false>(a);
}

}  // namespace fa2
