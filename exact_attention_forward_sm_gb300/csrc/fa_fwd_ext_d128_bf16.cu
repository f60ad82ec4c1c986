// Instantiations of the attention kernel with score variants (local window,
// soft cap, ALiBi) for head dim 128, bf16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_EXT_LAUNCHER(launch_ext_d128_bf16, 128, true)
}  // namespace fa
