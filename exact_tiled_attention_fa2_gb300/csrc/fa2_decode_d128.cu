// The tensor-core decode path for head dim 128 (every row count): the
// double-buffered kernel in split-key mode + the merge kernel, fp16 and bf16.
#include "fa2_decode_tc.cuh"

namespace fa2 {
int launch_decode_tc_d128(const LaunchArgs& a) { return launch_decode_tc<128>(a); }
}  // namespace fa2
