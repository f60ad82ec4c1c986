// Instantiations of the attention kernel for head dim 128, fp16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_LAUNCHER(launch_d128_fp16, 128, false)
}  // namespace fa
