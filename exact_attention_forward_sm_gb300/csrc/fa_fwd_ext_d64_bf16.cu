// Instantiations of the attention kernel with score variants (local window,
// soft cap, ALiBi) for head dim 64, bf16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_EXT_LAUNCHER(launch_ext_d64_bf16, 64, true)
}  // namespace fa
