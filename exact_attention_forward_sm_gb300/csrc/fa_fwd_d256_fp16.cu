// Instantiations of the head-dim-256 attention kernel, fp16.
#include "fa_fwd_wide.cuh"

namespace fa {
cudaError_t launch_d256_fp16(const LaunchArgs &a, bool causal, bool varlen) {
  if (causal)
    return varlen ? launch_wide<256, false, true, true, false>(a) : launch_wide<256, false, true, false, false>(a);
  return varlen ? launch_wide<256, false, false, true, false>(a) : launch_wide<256, false, false, false, false>(a);
}
}  // namespace fa
