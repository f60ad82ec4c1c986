// Instantiations of the head-dim-256 attention kernel with score variants
// (local window, soft cap, ALiBi, split-KV), fp16.
#include "fa_fwd_wide.cuh"

namespace fa {
cudaError_t launch_ext_d256_fp16(const LaunchArgs &a, bool varlen) {
  return varlen ? launch_wide<256, false, false, true, true>(a) : launch_wide<256, false, false, false, true>(a);
}
}  // namespace fa
