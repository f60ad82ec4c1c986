// Host-side launcher for one instantiation of the attention kernel.
#pragma once

#include <atomic>

#include "fa_fwd_kernel.cuh"

namespace fa {

struct LaunchArgs {
  CUtensorMap tm_q, tm_k, tm_v, tm_o;
  FwdParams p;
  int grid;
  cudaStream_t stream;
  int device;
};

template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool EXT = false, bool KVC = false>
cudaError_t launch_fwd(const LaunchArgs &a) {
  auto kern = fa_fwd_kernel<D, BF16, CAUSAL, VARLEN, EXT, KVC>;
  // opt in to the large dynamic shared memory once per device
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = 1ull << (a.device & 63);
  if (!(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)Smem<D, KVC>::kAlloc);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  kern<<<a.grid, kThreads, Smem<D, KVC>::kAlloc, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
  return cudaGetLastError();
}

// One translation unit per (head dim, dtype) instantiates the four
// (causal, packed) variants.
#define FA_DEFINE_LAUNCHER(NAME, D, BF16)                                       \
  cudaError_t NAME(const LaunchArgs &a, bool causal, bool varlen) {            \
    if (causal) {                                                               \
      return varlen ? launch_fwd<D, BF16, true, true>(a)                        \
                    : launch_fwd<D, BF16, true, false>(a);                      \
    }                                                                           \
    return varlen ? launch_fwd<D, BF16, false, true>(a)                         \
                  : launch_fwd<D, BF16, false, false>(a);                       \
  }

// Kernels with score variants (local window, soft cap, ALiBi): causal masking
// is folded into the window, so only the packed flag selects the instance.
#define FA_DEFINE_EXT_LAUNCHER(NAME, D, BF16)                                   \
  cudaError_t NAME(const LaunchArgs &a, bool varlen) {                         \
    return varlen ? launch_fwd<D, BF16, false, true, true>(a)                   \
                  : launch_fwd<D, BF16, false, false, true>(a);                 \
  }

// KV-cache decoding instances (score variants included).
#define FA_DEFINE_KVC_LAUNCHER(NAME, D, BF16)                                   \
  cudaError_t NAME(const LaunchArgs &a) { return launch_fwd<D, BF16, false, false, true, true>(a); }

cudaError_t launch_d64_fp16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d64_bf16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d128_fp16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d128_bf16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_ext_d64_fp16(const LaunchArgs &a, bool varlen);
cudaError_t launch_ext_d64_bf16(const LaunchArgs &a, bool varlen);
cudaError_t launch_ext_d128_fp16(const LaunchArgs &a, bool varlen);
cudaError_t launch_ext_d128_bf16(const LaunchArgs &a, bool varlen);
// Head dim 256 (one query tile per unit, see fa_fwd_wide.cuh).
cudaError_t launch_d256_fp16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d256_bf16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_ext_d256_fp16(const LaunchArgs &a, bool varlen);
cudaError_t launch_ext_d256_bf16(const LaunchArgs &a, bool varlen);
cudaError_t launch_kvc_d64_fp16(const LaunchArgs &a);
cudaError_t launch_kvc_d64_bf16(const LaunchArgs &a);
cudaError_t launch_kvc_d128_fp16(const LaunchArgs &a);
cudaError_t launch_kvc_d128_bf16(const LaunchArgs &a);

}  // namespace fa
