// fa2_decode_tc.cuh -- decoding on the tensor cores: the double-buffered
// forward kernel (fa2_fwd_dbuf.cuh) over (query tile, key chunk) units in
// split-key mode, then the decode merge kernel (fa2_decode.cuh) over the
// partials.  Used at d = 128 for any row count and at d = 64 from two rows
// on, where the score and value products outgrow the CUDA cores of the split
// decode kernel.
#pragma once

#include <cstring>

#include "fa2_decode.cuh"
#include "fa2_fwd_dbuf.cuh"

namespace fa2 {

template <int D, bool BF16, bool BAND>
int launch_decode_tc_kernels(const LaunchArgs& a) {
  if (a.p.splits <= 1) return launch_fwd_dbuf<D, BF16, BAND, false>(a);   // one chunk: O and LSE directly
  int e = launch_fwd_dbuf<D, BF16, BAND, true>(a);
  if (e != 0) return e;
  DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.f = a.p;
  dp.ws_o = a.p.ws_o;
  dp.ws_ml = a.p.ws_ml;
  dp.splits = a.p.splits;
  dp.chunk = a.p.split_chunk;
  dp.base = a.p.split_base;
  return launch_decode_merge<D, BF16>(dp, a.stream);
}

template <int D>
int launch_decode_tc(const LaunchArgs& a) {
  if (a.band) return a.bf16 ? launch_decode_tc_kernels<D, true, true>(a) : launch_decode_tc_kernels<D, false, true>(a);
  return a.bf16 ? launch_decode_tc_kernels<D, true, false>(a) : launch_decode_tc_kernels<D, false, false>(a);
}

}  // namespace fa2
