// Instantiations of the attention kernel for head dim 64, bf16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_LAUNCHER(launch_d64_bf16, 64, true)
}  // namespace fa
