// Fused exact attention forward for sm_103a (GB300): TMA + mbarrier pipeline,
// tcgen05 MMAs with TMEM accumulators, lazy-rescale online softmax.
//
// One CTA owns two 128-row query tiles that share every K/V tile it loads:
//   * grouped-query attention with an even group size: two query heads of one
//     K/V head, same rows (GQA head packing: each K/V tile serves both);
//   * otherwise: query rows [256 r, 256 r + 128) and [256 r + 128, 256 r + 256)
//     of one head.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3   softmax + epilogue for tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax + epilogue for tile 1
//   warp  8     TMEM allocation; lane 0 issues every tcgen05.mma
//   warp  9     lane 0 issues every TMA load
//   warps 10-11 idle
// After set-up the third warpgroup gives registers back (setmaxnreg) so the
// softmax warpgroups can hold a full 128-column score row: 2 x 128 x 208 +
// 128 x 56 = 60416 <= 384 x 168 registers granted at launch.
//
// Tensor memory (512 columns):  S0 [0,128)  S1 [128,256)  O0 [256,256+D)
// O1 [256+D, 256+2D).  P_t (16-bit pairs) overwrites columns [0,64) of S_t
// once the softmax has read S_t into registers, and is the A operand of
// O_t += P_t V taken straight from tensor memory.
//
// Per K/V tile j and query tile t the MMA warp issues, in this order,
//   O_t += P_t(j-1) V(j-1)   then   S_t = Q_t K(j)^T,
// and the tensor pipe executes one CTA's MMAs in issue order, so the S_t write
// of step j happens after the P_t read of step j-1 (the same ordering the
// pages' FA4 Blackwell kernel relies on for its S/P aliasing).
//
// Online softmax (release notes v1.7 section 1.2, v1.2 sections 1-2): row max
// m in raw score units, scale_log2 = scale * log2(e).  First K/V tile: m = its
// max.  Later tiles: scaled_diff = (m - max(m, tile max)) * scale_log2; if
// scaled_diff >= -threshold the rescale is skipped and m stays (max lagging),
// else row_sum and O_t are multiplied by exp2(scaled_diff) and m takes the new
// max.  P = exp2(s * scale_log2 - m * scale_log2) with the subtraction done by
// packed fma.rn.f32x2; m = -inf is treated as 0 (Check_inf).  The row sum adds
// the fp32 P before it is rounded to 16 bits for the PV product.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;      // query rows per tile
constexpr int kBlockN = 128;      // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr int kTmemCols = 512;
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 64 elements x 2 bytes

struct FwdParams {
  void *o;
  float *lse;
  const int32_t *cu_q;
  const int32_t *cu_k;
  int B, Hq, Hkv, Sq, Sk;   // packed problems: Sq / Sk are the packed totals
  int group;                // Hq / Hkv
  int pair_heads;           // 1: the two tiles are query heads 2u and 2u+1
  int head_units;           // head slots per sequence: Hq / 2 or Hq
  int rows_per_unit;        // query rows per CTA and head slot: 128 or 256
  int dense_row_units;      // dense problems: ceil(Sq / rows_per_unit)
  float scale_log2;         // scale * log2(e)
  float threshold;          // lazy-rescale threshold, log2 units
  long long wait_limit;     // bounded-wait limit in SM clock cycles
  int *status;              // device status word (first error wins)
};

template <int D>
struct Smem {
  static constexpr int kChunks = D / 64;                    // 64-element swizzle chunks
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
  static constexpr int kStages = (D == 128) ? 4 : 8;         // K/V ring depth
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = 2 * kTileBytes;
  static constexpr uint32_t kBarOff = kKVOff + kStages * kTileBytes;
  // barriers: q_full[2], kv_full[S], kv_empty[S], s_full[2], p_full[2], o_ready[2], drain
  static constexpr int kNumBars = 2 + 2 * kStages + 7;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kBytes = kMiscOff + 128;
  static constexpr uint32_t kAlloc = kBytes + 1024;  // slack for 1024-byte alignment
};

__device__ __forceinline__ void record_status(int *status, int code) { atomicCAS(status, 0, code); }

// Bounded wait on an mbarrier phase.  Gives up after `limit` cycles or, when
// `honor_abort` is set, as soon as another role raised the CTA abort flag; on
// a timeout records FA_ERR_TIMEOUT (value 4 of the C ABI) and raises the flag.
// Drains of in-flight copies / MMAs pass honor_abort = false so they still
// wait (bounded) for the hardware to finish before shared / tensor memory is
// released.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                         long long limit, int *status, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *abort_flag) return false;
    if (clock64() - t0 > limit) {
      record_status(status, 4);
      *abort_flag = 1;
      return false;
    }
  }
}

struct Work {
  int valid;
  int b, head[2], hkv;
  int m0[2];         // first query row of each tile within its sequence
  int lq, lk;        // sequence lengths
  int q_row0;        // tensor-map row of query row 0 of the sequence
  int k_row0;        // tensor-map row of key 0 of the sequence
  int map_b;         // tensor-map batch coordinate
  int64_t o_row0;    // global token index of query row 0 of the sequence
  int n_kv[2];       // K/V tiles each query tile visits
  int n_max;
};

template <bool CAUSAL>
__device__ __forceinline__ int tile_kv_count(int m0, int lq, int lk) {
  if (m0 >= lq || lk <= 0) return 0;
  const int full = (lk + kBlockN - 1) / kBlockN;
  if (!CAUSAL) return full;
  const int last_row = min(m0 + kBlockM, lq) - 1;
  const int last_key = last_row + lk - lq;  // bottom-right aligned diagonal
  if (last_key < 0) return 0;
  return min(full, last_key / kBlockN + 1);
}

// Decode this CTA's work unit.  Dense: row-unit index (heaviest causal rows
// first) is the slowest-varying part of blockIdx.x.  Packed: units are numbered
// sequence by sequence; warp 0 scans cu_seqlens cooperatively.
template <bool CAUSAL, bool VARLEN>
__device__ void decode_work(const FwdParams &p, Work &w, int lane) {
  w.valid = 0;
  const int unit = blockIdx.x;
  const int hu = unit % p.head_units;
  int b = 0, ru = 0, n_ru = 0;
  if (!VARLEN) {
    const int per_ru = p.B * p.head_units;
    ru = unit / per_ru;
    b = (unit % per_ru) / p.head_units;
    n_ru = p.dense_row_units;
    if (ru >= n_ru) return;
    w.lq = p.Sq;
    w.lk = p.Sk;
    w.q_row0 = 0;
    w.k_row0 = 0;
    w.map_b = b;
    w.o_row0 = (int64_t)b * p.Sq;
  } else {
    const int idx = unit / p.head_units;
    int base = 0, found = -1, found_ru = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int bb = b0 + lane;
      int cnt = 0;
      if (bb < p.B) {
        const int lq = p.cu_q[bb + 1] - p.cu_q[bb];
        cnt = lq > 0 ? (lq + p.rows_per_unit - 1) / p.rows_per_unit : 0;
      }
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += n;
      }
      const int excl = incl - cnt;
      const bool hit = bb < p.B && idx >= base + excl && idx < base + incl;
      const unsigned m = __ballot_sync(0xffffffffu, hit);
      if (m) {
        const int src = __ffs(m) - 1;
        found = b0 + src;
        found_ru = idx - base - __shfl_sync(0xffffffffu, excl, src);
        break;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (found < 0) return;
    b = found;
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    const int k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    if (q0 < 0 || q1 < q0 || q1 > p.Sq || k0 < 0 || k1 < k0 || k1 > p.Sk) {
      if (lane == 0) record_status(p.status, 5);
      return;
    }
    w.lq = q1 - q0;
    w.lk = k1 - k0;
    n_ru = (w.lq + p.rows_per_unit - 1) / p.rows_per_unit;
    ru = found_ru;
    w.q_row0 = q0;
    w.k_row0 = k0;
    w.map_b = 0;
    w.o_row0 = q0;
  }
  if (CAUSAL) ru = n_ru - 1 - ru;  // heavier (later) rows first
  w.b = b;
  if (p.pair_heads) {
    w.head[0] = 2 * hu;
    w.head[1] = 2 * hu + 1;
    w.m0[0] = w.m0[1] = ru * kBlockM;
  } else {
    w.head[0] = w.head[1] = hu;
    w.m0[0] = ru * 2 * kBlockM;
    w.m0[1] = ru * 2 * kBlockM + kBlockM;
  }
  w.hkv = w.head[0] / p.group;
  w.n_kv[0] = tile_kv_count<CAUSAL>(w.m0[0], w.lq, w.lk);
  w.n_kv[1] = tile_kv_count<CAUSAL>(w.m0[1], w.lq, w.lk);
  w.n_max = max(w.n_kv[0], w.n_kv[1]);
  w.valid = 1;
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Smem<D>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  auto q_full = [&](int t) { return bar0 + 8u * t; };
  auto kv_full = [&](int s) { return bar0 + 8u * (2 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (2 + L::kStages + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (2 + 2 * L::kStages + t); };
  auto p_full = [&](int t) { return bar0 + 8u * (4 + 2 * L::kStages + t); };
  auto o_ready = [&](int t) { return bar0 + 8u * (6 + 2 * L::kStages + t); };
  const uint32_t drain_bar = bar0 + 8u * (8 + 2 * L::kStages);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
  Work *work_s = reinterpret_cast<Work *>(smem + L::kMiscOff + 8);
  static_assert(sizeof(Work) <= 120, "work record does not fit");

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  if (warp == 0) {
    Work w;
    decode_work<CAUSAL, VARLEN>(p, w, lane);
    if (lane == 0) *work_s = w;
  }
  if (tid == 32) *abort_flag = 0;
  __syncthreads();
  const Work w = *work_s;
  if (!w.valid) return;

  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      mbar_init(q_full(t), 1);
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 4);
      mbar_init(o_ready(t), 1);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    mbar_init(drain_bar, 1);
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long limit = p.wait_limit;

  if (warp >= 8) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
  if (warp == kTmaWarp) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      int issued = 0;  // K/V loads issued (ring index)
      bool ok = true;
      for (int t = 0; t < 2; ++t) {
        if (w.n_kv[t] == 0) continue;
        mbar_arrive_expect_tx(q_full(t), L::kTileBytes);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_4d(sbase + L::kQOff + t * L::kTileBytes + c * kChunkBytes, &tm_q, q_full(t),
                      c * 64, w.head[t], w.q_row0 + w.m0[t], w.map_b, pol_q);
      }
      for (int j = 0; j < w.n_max && ok; ++j) {
        for (int which = 0; which < 2; ++which) {
          const int idx = 2 * j + which;
          const int s = idx % L::kStages;
          if (idx >= L::kStages &&
              !wait_bar(kv_empty(s), ((idx / L::kStages) + 1) & 1, abort_flag, limit, p.status)) {
            ok = false;
            break;
          }
          const CUtensorMap *tm = which == 0 ? &tm_k : &tm_v;
          mbar_arrive_expect_tx(kv_full(s), L::kTileBytes);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_4d(sbase + L::kKVOff + s * L::kTileBytes + c * kChunkBytes, tm, kv_full(s),
                        c * 64, w.hkv, w.k_row0 + j * kBlockN, w.map_b, pol_kv);
          issued = idx + 1;
        }
      }
      if (!ok) {
        // drain copies still in flight into the ring before the CTA exits
        for (int idx = max(0, issued - L::kStages); idx < issued; ++idx)
          wait_bar(kv_full(idx % L::kStages), (idx / L::kStages) & 1, abort_flag, limit, p.status,
                   false);
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0 && w.n_max > 0) {
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, kBlockM, D, true);
      bool ok = true;
      auto wait_kv = [&](int idx) {
        return wait_bar(kv_full(idx % L::kStages), (idx / L::kStages) & 1, abort_flag, limit, p.status);
      };
      auto issue_qk = [&](int t, int kidx) {
        const uint32_t qa = sbase + L::kQOff + t * L::kTileBytes;
        const uint32_t kb = sbase + L::kKVOff + (kidx % L::kStages) * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_ss(tmem + t * 128, make_sdesc_sw128(qa + off, 16, 1024),
                 make_sdesc_sw128(kb + off, 16, 1024), idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int vidx, bool first) {
        const uint32_t vb = sbase + L::kKVOff + (vidx % L::kStages) * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          mma_ts(tmem + 256 + t * D, tmem + t * 128 + kk * 8,
                 make_sdesc_sw128(vb + kk * 2048, kChunkBytes, 1024), idesc_pv,
                 (!first || kk > 0) ? 1u : 0u);
        }
      };
      // step 0: S_t = Q_t K(0)^T
      ok = wait_kv(0);
      for (int t = 0; t < 2 && ok; ++t) {
        if (w.n_kv[t] == 0) continue;
        ok = wait_bar(q_full(t), 0, abort_flag, limit, p.status);
        if (!ok) break;
        tc_fence_after();
        issue_qk(t, 0);
        tc_commit(s_full(t));
      }
      if (ok) tc_commit(kv_empty(0));
      for (int j = 1; j < w.n_max && ok; ++j) {
        const int kidx = 2 * j, vidx = 2 * j - 1;
        ok = wait_kv(kidx) && wait_kv(vidx);
        for (int t = 0; t < 2 && ok; ++t) {
          if (j - 1 < w.n_kv[t]) {
            ok = wait_bar(p_full(t), (j - 1) & 1, abort_flag, limit, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, vidx, j - 1 == 0);
            tc_commit(o_ready(t));
          }
          if (j < w.n_kv[t]) {
            issue_qk(t, kidx);
            tc_commit(s_full(t));
          }
        }
        if (ok) {
          tc_commit(kv_empty(vidx % L::kStages));
          tc_commit(kv_empty(kidx % L::kStages));
        }
      }
      if (ok) {
        const int j = w.n_max;
        const int vidx = 2 * j - 1;
        ok = wait_kv(vidx);
        for (int t = 0; t < 2 && ok; ++t) {
          if (j - 1 < w.n_kv[t]) {
            ok = wait_bar(p_full(t), (j - 1) & 1, abort_flag, limit, p.status);
            if (!ok) break;
            tc_fence_after();
            issue_pv(t, vidx, j - 1 == 0);
            tc_commit(o_ready(t));
          }
        }
        if (ok) tc_commit(kv_empty(vidx % L::kStages));
      }
      // make sure no MMA is still running when tensor memory is released
      tc_commit(drain_bar);
      wait_bar(drain_bar, 0, abort_flag, limit, p.status, false);
    }
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 208;" ::: "memory");
    // ------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;        // query tile of this warpgroup
    const int quarter = warp & 3;   // TMEM lane quarter
    const int row = quarter * 32 + lane;
    const int qi = w.m0[t] + row;   // query row within its sequence
    const int n_kv = w.n_kv[t];
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_addr = lane_base + t * 128;
    const uint32_t o_addr = lane_base + 256 + t * D;
    const float scale_log2 = p.scale_log2;
    const float neg_thr = -p.threshold;
    const int diag = qi + w.lk - w.lq;  // last visible key of this row (causal)
    // every lane of a warp must agree before the warp-wide tcgen05.ld / st
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
      const bool got = wait_bar(bar, parity, abort_flag, limit, p.status);
      return __all_sync(0xffffffffu, got);
    };
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      if (!warp_wait(s_full(t), j & 1)) { ok = false; break; }
      tc_fence_after();
      uint32_t sr[128];
      tmem_ld128_wait(s_addr, sr);
      float *s = reinterpret_cast<float *>(sr);
      const int k0 = j * kBlockN;
      const bool need_mask =
          (k0 + kBlockN > w.lk) || (CAUSAL && (k0 + kBlockN - 1 > w.m0[t] + w.lk - w.lq));
      if (need_mask) {
        int lim = w.lk - k0;
        if (CAUSAL) lim = min(lim, diag - k0 + 1);
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
      }
      float bm = s[0];
#pragma unroll
      for (int c = 1; c < kBlockN; ++c) bm = fmaxf(bm, s[c]);
      float alpha = 1.f;
      bool rescale = false;
      if (j == 0) {
        m = bm;
      } else {
        const float m_cur = fmaxf(m, bm);
        const float diff = (m_cur == -INFINITY) ? 0.f : (m - m_cur) * scale_log2;
        if (!(diff >= neg_thr)) {
          alpha = ex2(diff);
          l *= alpha;
          m = m_cur;
          rescale = true;
        }
      }
      if (__any_sync(0xffffffffu, rescale)) {
        // O_t(j-1) must be final before it is rescaled in place
        if (!warp_wait(o_ready(t), (j - 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t orr[32];
          tmem_ld32_wait(o_addr + c * 32, orr);
#pragma unroll
          for (int i = 0; i < 32; ++i) orr[i] = __float_as_uint(__uint_as_float(orr[i]) * alpha);
          tmem_st32(o_addr + c * 32, orr);
        }
      }
      const float ms = (m == -INFINITY) ? 0.f : m * scale_log2;
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c4 * 32 + 2 * i;
          float x0, x1;
          fma_f32x2(x0, x1, s[c], s[c + 1], scale_log2, scale_log2, -ms, -ms);
          const float p0 = ex2(x0), p1 = ex2(x1);
          ls0 += p0;
          ls1 += p1;
          if (BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);
            pk[i] = *reinterpret_cast<uint32_t *>(&h);
          } else {
            __half2 h = __floats2half2_rn(p0, p1);
            pk[i] = *reinterpret_cast<uint32_t *>(&h);
          }
        }
        tmem_st16(s_addr + c4 * 16, pk);  // 32 keys -> 16 packed columns
      }
      l += ls0 + ls1;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(t));
    }
    // --------------------------------------------------------------- epilogue
    const bool row_valid = qi < w.lq && w.m0[t] < w.lq;
    const int64_t tok = w.o_row0 + qi;
    if (ok && w.m0[t] < w.lq) {
      elem_t *o = reinterpret_cast<elem_t *>(p.o) + (tok * p.Hq + w.head[t]) * (int64_t)D;
      if (n_kv > 0) {
        if (warp_wait(o_ready(t), (n_kv - 1) & 1)) {
          tc_fence_after();
          const float inv_l = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32_wait(o_addr + c * 32, orr);
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = __uint_as_float(orr[2 * i]) * inv_l;
              const float b = __uint_as_float(orr[2 * i + 1]) * inv_l;
              if (BF16) {
                __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                pk[i] = *reinterpret_cast<uint32_t *>(&h);
              } else {
                __half2 h = __floats2half2_rn(a, b);
                pk[i] = *reinterpret_cast<uint32_t *>(&h);
              }
            }
            if (row_valid) {
              uint4 *dst = reinterpret_cast<uint4 *>(o + c * 32);
#pragma unroll
              for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
          }
        } else {
          ok = false;
        }
      } else if (row_valid) {
        uint4 *dst = reinterpret_cast<uint4 *>(o);
#pragma unroll
        for (int i = 0; i < D / 8; ++i) dst[i] = make_uint4(0, 0, 0, 0);
      }
      if (ok && row_valid && p.lse != nullptr) {
        const float lse = (l > 0.f) ? (m * scale_log2 + log2f(l)) * 0.69314718055994531f
                                    : -INFINITY;
        const int64_t li = VARLEN ? (int64_t)w.head[t] * p.Sq + tok
                                  : ((int64_t)w.b * p.Hq + w.head[t]) * p.Sq + qi;
        p.lse[li] = lse;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace fa
