// Split-KV combine kernel: host-side interface.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

struct CombineParams {
  const float *o_part;    // [num_splits][rows][D] fp32, normalised O of each split
  const float *lse_part;  // [num_splits][rows] fp32, LSE of each split (-inf: empty)
  void *o;                // output, layout of the forward call (16-bit)
  float *lse;             // output LSE (LSE-index order) or null
  int64_t rows;           // LSE entries: dense B * Hq * Sq, packed Hq * Sq
  int num_splits;
  int B, Hq, Sq;          // packed problems: Sq = total query tokens
  const int32_t *cu_q;    // packed: cu_seqlens_q (device), else null
};

cudaError_t launch_combine(const CombineParams &p, int D, bool bf16, int sms,
                           cudaStream_t stream);

}  // namespace fa
