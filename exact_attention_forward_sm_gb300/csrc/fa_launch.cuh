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

// Generation of the per-device launch state (defined in fa_api.cu).
// fa_shutdown() advances it, so every kernel sets its shared-memory attribute
// again on its next launch on each device.
std::atomic<unsigned> &launch_epoch();

// A kernel's opt-in to its large dynamic shared memory, made once per device
// and epoch: `bits` has bit (device % 64) set once the attribute is set.  The
// same first launch checks that the kernel was built with `regs` registers
// per thread: its warp roles trade registers with setmaxnreg on the basis of
// that launch count, and a different count would leave a role waiting for
// registers that never come free, so such a build is refused instead.
struct SmemOptIn {
  std::atomic<unsigned long long> bits{0};
  std::atomic<unsigned> epoch{0};

  template <class Kernel>
  cudaError_t ensure(Kernel kern, int bytes, int device, int regs) {
    const unsigned ep = launch_epoch().load(std::memory_order_acquire);
    if (epoch.load(std::memory_order_acquire) != ep) {
      bits.store(0, std::memory_order_release);
      epoch.store(ep, std::memory_order_release);
    }
    const unsigned long long bit = 1ull << (device & 63);
    if (bits.load(std::memory_order_acquire) & bit) return cudaSuccess;
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kern);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != regs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) bits.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }
};

template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool EXT = false, bool KVC = false,
          int VAR = kVarCap | kVarAlibi>
cudaError_t launch_fwd(const LaunchArgs &a) {
  auto kern = fa_fwd_kernel<D, BF16, CAUSAL, VARLEN, EXT, KVC, VAR>;
  static SmemOptIn opt_in;
  const cudaError_t e = opt_in.ensure(kern, (int)Smem<D, KVC, VARLEN || KVC>::kAlloc, a.device, 65536 / kThreads / 8 * 8);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, kThreads, Smem<D, KVC, VARLEN || KVC>::kAlloc, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_o, a.p);
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

// Kernels with score variants (local window, split-KV, soft cap, ALiBi):
// causal masking is folded into the window; the packed flag and the variants
// that are on (kVarCap / kVarAlibi bits) select the instance.
#define FA_EXT_INSTANCE(D, BF16, VAR)                                           \
  (varlen ? launch_fwd<D, BF16, false, true, true, false, VAR>(a)               \
          : launch_fwd<D, BF16, false, false, true, false, VAR>(a))
#define FA_DEFINE_EXT_LAUNCHER(NAME, D, BF16)                                   \
  cudaError_t NAME(const LaunchArgs &a, bool varlen, int var) {                \
    switch (var) {                                                              \
      case 0: return FA_EXT_INSTANCE(D, BF16, 0);                               \
      case kVarCap: return FA_EXT_INSTANCE(D, BF16, kVarCap);                   \
      case kVarAlibi: return FA_EXT_INSTANCE(D, BF16, kVarAlibi);               \
      default: return FA_EXT_INSTANCE(D, BF16, kVarCap | kVarAlibi);            \
    }                                                                           \
  }

// KV-cache decoding instances (score variants included).
#define FA_DEFINE_KVC_LAUNCHER(NAME, D, BF16)                                   \
  cudaError_t NAME(const LaunchArgs &a) { return launch_fwd<D, BF16, false, false, true, true>(a); }

cudaError_t launch_d64_fp16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d64_bf16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d128_fp16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_d128_bf16(const LaunchArgs &a, bool causal, bool varlen);
cudaError_t launch_ext_d64_fp16(const LaunchArgs &a, bool varlen, int var);
cudaError_t launch_ext_d64_bf16(const LaunchArgs &a, bool varlen, int var);
cudaError_t launch_ext_d128_fp16(const LaunchArgs &a, bool varlen, int var);
cudaError_t launch_ext_d128_bf16(const LaunchArgs &a, bool varlen, int var);
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
