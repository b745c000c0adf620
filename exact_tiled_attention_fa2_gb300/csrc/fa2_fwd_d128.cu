// Forward kernel instantiations for head dim 128: one 128-row query tile per
// CTA, 64-row key/value tiles, two S buffers in tensor memory, two CTAs per SM.
#include "fa2_fwd_dbuf.cuh"

namespace fa2 {
int launch_fwd_d128(const LaunchArgs& a) { return launch_fwd_dbuf_dispatch<128>(a); }
}  // namespace fa2
