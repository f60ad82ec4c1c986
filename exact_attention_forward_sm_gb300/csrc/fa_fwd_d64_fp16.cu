// Instantiations of the attention kernel for head dim 64, fp16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_LAUNCHER(launch_d64_fp16, 64, false)
}  // namespace fa
