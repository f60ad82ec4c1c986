// Instantiations of the head-dim-256 attention kernel with score variants
// (local window, soft cap, ALiBi, split-KV), bf16.
#include "fa_fwd_wide.cuh"

namespace fa {
cudaError_t launch_ext_d256_bf16(const LaunchArgs &a, bool varlen) {
  return varlen ? launch_wide<256, true, false, true, true>(a) : launch_wide<256, true, false, false, true>(a);
}
}  // namespace fa
