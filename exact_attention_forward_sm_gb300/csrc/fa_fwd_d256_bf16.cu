// Instantiations of the head-dim-256 attention kernel, bf16.
#include "fa_fwd_wide.cuh"

namespace fa {
cudaError_t launch_d256_bf16(const LaunchArgs &a, bool causal, bool varlen) {
  if (causal)
    return varlen ? launch_wide<256, true, true, true, false>(a) : launch_wide<256, true, true, false, false>(a);
  return varlen ? launch_wide<256, true, false, true, false>(a) : launch_wide<256, true, false, false, false>(a);
}
}  // namespace fa
