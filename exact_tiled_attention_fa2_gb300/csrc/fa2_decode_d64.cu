// Decode kernel instantiations for head dim 64 (1, 2, 4 or 8 query rows, fp16 and bf16),
// and the tensor-core decode path (double-buffered kernel in split-key mode + merge).
#include "fa2_decode_tc.cuh"

namespace fa2 {
int launch_decode_d64(const DecodeLaunchArgs& a) { return launch_decode_dispatch<64>(a); }
int launch_decode_tc_d64(const LaunchArgs& a) { return launch_decode_tc<64>(a); }
}  // namespace fa2
