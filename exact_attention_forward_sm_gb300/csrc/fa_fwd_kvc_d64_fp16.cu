// Instantiations of the attention kernel for KV-cache decoding (paged or
// contiguous cache, packed GQA heads) for head dim 64, fp16.
#include "fa_launch.cuh"

namespace fa {
FA_DEFINE_KVC_LAUNCHER(launch_kvc_d64_fp16, 64, false)
}  // namespace fa
