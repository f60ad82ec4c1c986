// Split-KV combine: merges the per-split partial results of the attention
// kernel (normalised fp32 O_s and LSE_s of each K/V chunk) into O and LSE.
// Split-KV forward with an LSE-weighted merge is the upstream FA2 kvcache /
// split path that the fork's v1.2 notes, section 3, list among the dispatch
// sites (compute_attn_1rowblock_splitkv).
//
// For one row with splits s = 1..S:  M = max_s LSE_s,  w_s = exp(LSE_s - M),
//   O = sum_s w_s O_s / sum_s w_s,   LSE = M + ln sum_s w_s;
// a split that saw no visible key has LSE_s = -inf and weight 0, and a row no
// split saw gets O = 0, LSE = -inf.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "fa_combine.cuh"
#include "fa_ptx.cuh"

namespace fa {

namespace {

template <int N, bool BF16>
__device__ __forceinline__ void store_row(void *dst, const float (&x)[N]) {
  static_assert(N == 2 || N == 4 || N == 8, "values per lane");
  uint32_t w[N / 2];
#pragma unroll
  for (int k = 0; k < N / 2; ++k) {
    if constexpr (BF16) {
      __nv_bfloat162 h = __floats2bfloat162_rn(x[2 * k], x[2 * k + 1]);
      w[k] = *reinterpret_cast<uint32_t *>(&h);
    } else {
      __half2 h = __floats2half2_rn(x[2 * k], x[2 * k + 1]);
      w[k] = *reinterpret_cast<uint32_t *>(&h);
    }
  }
  if constexpr (N == 8)
    *reinterpret_cast<uint4 *>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
  else if constexpr (N == 4)
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[1]);
  else
    *reinterpret_cast<uint32_t *>(dst) = w[0];
}

// One warp per row (LSE-index order); lane l owns columns [l N, l N + N).
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_combine_kernel(const CombineParams p) {
  constexpr int N = D / 32;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  int tok_lo = 0, tok_hi = p.Sq;
  if (p.cu_q) {  // packed: only tokens of some sequence were computed
    tok_lo = max(0, p.cu_q[0]);
    tok_hi = min(p.Sq, p.cu_q[p.B]);
  }
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < p.rows;
       r += warps) {
    int64_t o_row;  // row of O ([tokens, Hq] order)
    if (p.cu_q) {
      const int64_t h = r / p.Sq, tok = r % p.Sq;
      if (tok < tok_lo || tok >= tok_hi) continue;
      o_row = tok * p.Hq + h;
    } else {
      const int64_t per_b = (int64_t)p.Hq * p.Sq;
      const int64_t b = r / per_b, h = (r / p.Sq) % p.Hq, i = r % p.Sq;
      o_row = (b * p.Sq + i) * p.Hq + h;
    }
    float m = -INFINITY;
    for (int s = lane; s < p.num_splits; s += 32) m = fmaxf(m, p.lse_part[s * p.rows + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float acc[N];
#pragma unroll
    for (int k = 0; k < N; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < p.num_splits; ++s) {
        const float w = ex2((p.lse_part[s * p.rows + r] - m) * 1.4426950408889634f);
        wsum += w;
        const float *src = p.o_part + (s * p.rows + r) * D + lane * N;
        if constexpr (N == 8) {
          const float4 x = *reinterpret_cast<const float4 *>(src);
          const float4 y = *reinterpret_cast<const float4 *>(src + 4);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
          acc[2] = fmaf(w, x.z, acc[2]);
          acc[3] = fmaf(w, x.w, acc[3]);
          acc[4] = fmaf(w, y.x, acc[4]);
          acc[5] = fmaf(w, y.y, acc[5]);
          acc[6] = fmaf(w, y.z, acc[6]);
          acc[7] = fmaf(w, y.w, acc[7]);
        } else if constexpr (N == 4) {
          const float4 x = *reinterpret_cast<const float4 *>(src);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
          acc[2] = fmaf(w, x.z, acc[2]);
          acc[3] = fmaf(w, x.w, acc[3]);
        } else {
          const float2 x = *reinterpret_cast<const float2 *>(src);
          acc[0] = fmaf(w, x.x, acc[0]);
          acc[1] = fmaf(w, x.y, acc[1]);
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int k = 0; k < N; ++k) acc[k] *= inv;
    store_row<N, BF16>(reinterpret_cast<elem_t *>(p.o) + o_row * D + lane * N, acc);
    if (lane == 0 && p.lse) p.lse[r] = wsum > 0.f ? m + logf(wsum) : -INFINITY;
  }
}

}  // namespace

cudaError_t launch_combine(const CombineParams &p, int D, bool bf16, int sms,
                           cudaStream_t stream) {
  constexpr int kWarps = 8;
  int64_t blocks = (p.rows + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 1) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  const dim3 grid((unsigned)blocks), block(32 * kWarps);
  if (D == 64) {
    if (bf16)
      fa_combine_kernel<64, true><<<grid, block, 0, stream>>>(p);
    else
      fa_combine_kernel<64, false><<<grid, block, 0, stream>>>(p);
  } else if (D == 256) {
    if (bf16)
      fa_combine_kernel<256, true><<<grid, block, 0, stream>>>(p);
    else
      fa_combine_kernel<256, false><<<grid, block, 0, stream>>>(p);
  } else {
    if (bf16)
      fa_combine_kernel<128, true><<<grid, block, 0, stream>>>(p);
    else
      fa_combine_kernel<128, false><<<grid, block, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace fa
