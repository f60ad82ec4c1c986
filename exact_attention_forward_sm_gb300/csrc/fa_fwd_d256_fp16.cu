// Instantiations of the head-dim-256 attention kernel, fp16.
#include "fa_fwd_wide.cuh"

namespace fa {
cudaError_t launch_d256_fp16(const LaunchArgs &a, bool causal, bool varlen) {
  if (causal)
    return varlen ? launch_wide<false, true, true, false>(a) : launch_wide<false, true, false, false>(a);
  return varlen ? launch_wide<false, false, true, false>(a) : launch_wide<false, false, false, false>(a);
}
}  // namespace fa
