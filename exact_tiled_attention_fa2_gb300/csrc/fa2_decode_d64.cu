// Decode kernel instantiations for head dim 64 (1, 2, 4 or 8 query rows, fp16 and bf16).
#include "fa2_decode.cuh"

namespace fa2 {
int launch_decode_d64(const DecodeLaunchArgs& a) { return launch_decode_dispatch<64>(a); }
}  // namespace fa2
