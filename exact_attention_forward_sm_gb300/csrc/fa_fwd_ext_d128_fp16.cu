// Instantiations of the attention kernel with score variants (local window,
// soft cap, ALiBi) for head dim 128, fp16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_EXT_LAUNCHER(launch_ext_d128_fp16, 128, false)
}  // namespace fa
