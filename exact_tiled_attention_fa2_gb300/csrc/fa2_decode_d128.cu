// Decode kernel instantiations for head dim 128 (1, 2, 4 or 8 query rows, fp16 and bf16),
// and the tensor-core decode path (double-buffered kernel in split-key mode + merge).
#include "fa2_decode_tc.cuh"

namespace fa2 {
int launch_decode_d128(const DecodeLaunchArgs& a) { return launch_decode_dispatch<128>(a); }
int launch_decode_tc_d128(const LaunchArgs& a) { return launch_decode_tc<128>(a); }
}  // namespace fa2
