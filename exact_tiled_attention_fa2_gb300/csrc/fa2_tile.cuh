// fa2_tile.cuh -- pieces the tiled tensor-core kernels share: the online
// softmax's rescaling margin, the max of three, K-major descriptor steps and
// the exponentiation of one 32-column chunk of S into 16-bit P in TMEM.
#pragma once

#include "fa2_common.cuh"

namespace fa2 {

// The running maximum is only raised when a key tile's maximum exceeds it by
// more than kRescaleLog2 (2^8): otherwise P = 2^(s - m) may reach 2^8, which
// 16-bit P and fp32 l and O~ hold as exactly as values below 1, and O~ need
// not be rescaled.  The result is the same exact softmax: every term and l
// use the same m, and LSE = (m + log2 l) ln 2.  (Deferred normalisation taken
// one step further than FlashAttention V2 in depth, section 3.2.)
constexpr float kRescaleLog2 = 8.0f;

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Shared-memory descriptors are built once and advanced by adding (byte
// offset >> 4) to the start-address field: every tile sits below 256 KB of
// shared memory, so the 14-bit field never carries into the next one.  Step
// k (16 columns of a K-major, 128-byte-swizzled operand of `rows` rows) lies
// in 64-column block k / 4, 32 bytes per step inside it.
template <class C>
__device__ __forceinline__ constexpr uint64_t kmajor_step(int k, int rows) {
  return (uint64_t)(((k >> 2) * (rows * 128) + (k & 3) * 32) >> 4);
}

// Exponentiate one 32-column chunk of S (exp2 domain: 2^(s * scale_log2 - m))
// into packed 16-bit P (and, when SPLIT, its low part P - P_hi) and store it
// to the chunk's TMEM columns; the row sums go to sum0 / sum1.
template <class C, bool BF16, bool SPLIT>
__device__ __forceinline__ void softmax_p_chunk(const uint32_t* sr, int ch, uint32_t tS, float2 scale2, float2 neg_m2,
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

}  // namespace fa2
