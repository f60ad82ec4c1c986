// Instantiations of the attention kernel for head dim 128, bf16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_LAUNCHER(launch_d128_bf16, 128, true)
}  // namespace fa
