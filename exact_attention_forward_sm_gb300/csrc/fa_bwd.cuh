// Backward pass of exact attention (dQ, dK, dV) for sm_103a: declarations
// shared by the C ABI and the kernels in fa_bwd.cu.
//
// The gradients of softmax attention, per query row with its visible keys
// (P = softmax(scale Q K^T), dP = dO V^T, Delta = rowsum(dO * O)):
//   dS = P * (dP - Delta),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO.
// The fork's v1.7 release notes validate such a backward pass (section 4.4).
// Three launches: a row pass (Delta and the LSE in log2 units), a key-tile
// pass (dK, dV accumulated in tensor memory over every query tile and every
// query head of the K/V head's group) and a query-tile pass (dQ accumulated
// over the visible key tiles).  Every output element is written exactly once,
// so the result is deterministic.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace fa {

struct BwdParams {
  const void *o;       // forward output [B, Sq, Hq, D] (16-bit)
  const void *dout;    // upstream gradient, same layout
  const float *lse;    // forward LSE [B, Hq, Sq] (natural log)
  float *lse_l2;       // workspace: LSE * log2(e), +inf for rows without keys
  float *delta;        // workspace: rowsum(dO * O) in fp32
  void *dq, *dk, *dv;  // outputs, layouts of q, k, v
  const int32_t *cu_q, *cu_k;  // packed sequences: B + 1 offsets each (else null)
  int B, Hq, Hkv, Sq, Sk, group;  // packed: B sequences, Sq / Sk the packed totals
  float scale, scale_log2;
  int q_tiles, k_tiles;
  long long wait_limit;  // bounded-wait limit in cycles
  int *status;           // device status word (FA_ERR_TIMEOUT on a timeout)
};

struct BwdLaunch {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  BwdParams p;
  cudaStream_t stream;
  int device;
  int sms;  // SM count of the device (persistent grids)
};

// Launches the three passes for head dim 64 or 128 (bf16 or fp16), dense or
// packed (p.cu_q / p.cu_k set).
cudaError_t launch_bwd(const BwdLaunch &a, int D, bool bf16, bool causal, bool varlen);

}  // namespace fa
