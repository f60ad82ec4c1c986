// Fused exact attention forward for sm_103a (GB300): persistent CTAs, TMA +
// mbarrier pipeline, tcgen05 MMAs with TMEM accumulators, lazy-rescale online
// softmax.
//
// Work unit: two 128-row query tiles that share every K/V tile loaded for them:
//   * grouped-query attention with an even group size: two query heads of one
//     K/V head, same rows (GQA head packing: each K/V tile serves both);
//   * otherwise: query rows [256 r, 256 r + 128) and [256 r + 128, 256 r + 256)
//     of one head.
// Units are numbered heaviest first (causal: last row blocks first).  The grid
// has at most one CTA per SM; CTA b takes units b, 2G-1-b, 2G+b, 4G-1-b, ...
// (G = grid size): a snake over the heavy-first order, which balances causal
// problems like a greedy longest-first schedule without any global counter.
// Barriers, tensor memory and the K/V ring live across units, so one unit's
// epilogue overlaps the next unit's loads and first Q K^T.
//
// Warp roles (384 threads, three warpgroups):
//   warps 0-3   softmax + epilogue for tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax + epilogue for tile 1
//   warp  8     TMEM allocation; lane 0 issues tile 0's tcgen05.mma
//   warp  9     lane 0 issues every TMA load
//   warp  10    lane 0 issues tile 1's tcgen05.mma
//   warp  11    zeroes the V rows past a sequence's last key in the last K/V
//               tile of a unit (packed sequences, KV caches), where the tile
//               reads other data
// After set-up the third warpgroup gives registers back (setmaxnreg) so the
// softmax warpgroups can hold a full 128-column score row: 2 x 128 x 192 +
// 128 x 96 = 61440 <= 384 x 168 registers granted at launch.
//
// Tensor memory (512 columns):  S0 [0,128)  S1 [128,256)  O0 [256,256+D)
// O1 [256+D, 256+2D).  P_t (16-bit pairs) overwrites columns [0,64) of S_t
// once the softmax has read S_t into registers, and is the A operand of
// O_t += P_t V taken straight from tensor memory.
//
// Per K/V tile j and query tile t the MMA thread issues, in this order,
//   O_t += P_t(j-1) V(j-1)   then   S_t = Q_t K(j)^T,
// with the first half of O += P V (keys 0-63) started as soon as the softmax
// has stored those P values, while it still computes keys 64-127;
// alternating tiles, so tile 0's softmax runs while the tensor pipe works on
// tile 1 and vice versa.  The tensor pipe executes one CTA's MMAs in issue
// order, so the S_t write of step j happens after the P_t read of step j-1
// (the ordering upstream's FA4 Blackwell kernel relies on for its S/P
// aliasing, per the upstream code survey's FA4 section and the FA4
// changelog's S/P ping-pong note).  Descriptors are built once and each MMA adds a compile-time
// offset: the tensor pipe's MMA queue is about one instruction deep, so the
// issuing thread must emit the next MMA as soon as one starts, and the issue
// stream is kept branch-free.  For the same reason the issuers poll the P
// barriers and the turn flag instead of suspending on them (a suspended thread
// wakes ~200 cycles after the phase completes).
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
#include <type_traits>

#include "fa_ptx.cuh"

namespace fa {

constexpr int kBlockM = 128;      // query rows per tile
constexpr int kBlockN = 128;      // keys per K/V tile
constexpr int kThreads = 384;
constexpr int kMmaWarp = 8;   // issues tile 0's MMAs (and owns the TMEM allocation)
constexpr int kTmaWarp = 9;
constexpr int kMmaWarp2 = 10; // issues tile 1's MMAs
constexpr int kFixWarp = 11;  // zeroes V rows past a sequence's keys
constexpr int kTmemCols = 512;
constexpr uint32_t kChunkBytes = 128 * 128;  // 128 rows x 64 elements x 2 bytes

// n / d for 0 <= n < 2^31 as a multiply-high and a shift (Granlund and
// Montgomery's division by invariant integers, round-up reciprocal): with
// p = 31 + ceil(log2 d) and m = ceil(2^p / d) < 2^32, the error of n m / 2^p
// against n / d is below 2^(31 - p) <= 1 / d, which never reaches the next
// integer, so floor(n / d) = floor(n m / 2^p).  d = 1 passes n through.
struct FastDiv {
  int d;
  uint32_t mul;
  uint32_t shift;  // p - 32
};

inline FastDiv make_fast_div(int d) {
  FastDiv f{d, 0u, 0u};
  if (d > 1) {
    int l = 0;
    while ((1ll << l) < d) ++l;
    const int p = 31 + l;
    f.mul = (uint32_t)(((1ull << p) + (uint64_t)d - 1) / (uint64_t)d);
    f.shift = (uint32_t)(p - 32);
  }
  return f;
}

__device__ __forceinline__ int fast_div(const FastDiv &f, int n) {
  return f.d == 1 ? n : (int)(__umulhi((uint32_t)n, f.mul) >> f.shift);
}

struct FwdParams {
  void *o;
  float *lse;
  const int32_t *cu_q;
  const int32_t *cu_k;
  int B, Hq, Hkv, Sq, Sk;   // packed problems: Sq / Sk are the packed totals
  int group;                // Hq / Hkv
  int pair_heads;           // 1: the two tiles are query heads 2u and 2u+1
  int head_units;           // head slots per sequence: Hq / 2 or Hq
  int rows_per_unit;        // query rows per unit and head slot: 128 or 256
  int dense_row_units;      // dense problems: ceil(Sq / rows_per_unit)
  int rows_fastest;         // dense, every unit the same work (no causal mask, no
                            // window): the row unit varies fastest, so the
                            // CTAs running together share one head's K / V in L2
  int total_units;          // units to process (packed: an upper bound)
  float scale_log2;         // scale * log2(e)
  float threshold;          // lazy-rescale threshold, log2 units
  // score variants (kernels instantiated with EXT only)
  int win_l, win_r;         // local window around the diagonal, -1 = unbounded;
                            // a causal mask arrives here as win_r = 0
  int reverse_rows;         // later row blocks see more keys: schedule them first
  float cap_k;              // soft cap c: scale / c, 0 = no soft cap
  float cap_l2;             // soft cap c: c * log2(e)
  const float *alibi;       // ALiBi slope per query head (natural-log units) or null
  // split-KV (instances with score variants only): each unit of the problem
  // becomes num_splits units, split s taking the s-th of num_splits equal
  // chunks of its sequence's K/V tiles and writing a partial result instead
  // of O / LSE
  int num_splits;           // 1: no split (o_part / lse_part unused)
  float *o_part;            // [num_splits][part_rows][D] fp32, O_s / l_s
  float *lse_part;          // [num_splits][part_rows] fp32, LSE_s (-inf: no visible key)
  int64_t part_rows;        // rows per split slab: one per LSE entry
  // KV-cache decoding (instances with KVC): q / o dense [B, Sq, Hq, D]; the
  // keys of sequence b are its first cache_seqlens[b] cache rows, key j being
  // row j % page_rows of page block_table[b * max_blocks + j / page_rows]
  // (page b when there is no table).  A tile packs the `group` query heads of
  // one K/V head for tok_per_tile = 128 / group consecutive tokens (row r:
  // token r / group, head r % group), and both tiles of a unit hold the same
  // rows and split its K/V tiles between them (even / odd); their partial
  // results are merged in the epilogue.
  const int32_t *cache_seqlens;
  const int32_t *block_table;
  int max_blocks;           // block_table row length
  int page_rows;            // cache rows per page
  int num_pages;            // pages in the cache
  int tok_per_tile;         // 128 / group
  int tok_blocks;           // ceil(Sq / tok_per_tile)
  // the divisors of the unit index, set by set_divisors() once the fields
  // above are final
  FastDiv div_splits, div_head_units, div_B, div_Hkv, div_tok_blocks, div_ru;
  long long wait_limit;     // bounded-wait limit in SM clock cycles
  int *status;              // device status word (first error wins)
  unsigned long long *trace;  // clock64 pipeline trace (trace builds only)
};

inline void set_divisors(FwdParams &p) {
  p.div_splits = make_fast_div(p.num_splits > 1 ? p.num_splits : 1);
  p.div_head_units = make_fast_div(p.head_units > 0 ? p.head_units : 1);
  p.div_B = make_fast_div(p.B > 0 ? p.B : 1);
  p.div_Hkv = make_fast_div(p.Hkv > 0 ? p.Hkv : 1);
  p.div_tok_blocks = make_fast_div(p.tok_blocks > 0 ? p.tok_blocks : 1);
  p.div_ru = make_fast_div(p.dense_row_units > 0 ? p.dense_row_units : 1);
}

// Pipeline trace (compiled in with -DFA_TRACE): CTA 0 records SM clock stamps
// of the K/V steps of its first unit into a 2048-entry buffer.
//   softmax tile t, step j < 63:  (t * 64 + j) * 8 + e   e: 0 S ready, 1 S in
//       registers, 2 max / rescale decided, 3 P of keys 0-63 signalled, 4 P of
//       keys 64-127 signalled; (t * 64 + 63) * 8 + 5 / 6: epilogue start / end
//   MMA issuer of tile t, step j:  1024 + j * 8 + 2 + 2t + e   e: 0 inputs
//       ready, 1 O_t += P_t(j-1) V(j-1) and S_t = Q_t K(j)^T issued
//   TMA load idx < 256:           1536 + idx  (issue time)
//   2047: kernel start
constexpr int kTraceEntries = 2048;
#ifdef FA_TRACE
#define FA_TRACE_AT(cond, idx)                                               \
  do {                                                                       \
    if ((cond) && blockIdx.x == 0 && p.trace) p.trace[(idx)] = clock64();    \
  } while (0)
#else
#define FA_TRACE_AT(cond, idx) \
  do {                         \
  } while (0)
#endif

// FIX: the kernel reads K/V tiles that may reach past a sequence's keys into
// other data (packed sequences, KV caches) and carries the v_fixed barriers.
template <int D, bool KVC = false, bool FIX = false>
struct Smem {
  static constexpr int kChunks = D / 64;                    // 64-element swizzle chunks
  static constexpr uint32_t kTileBytes = kChunks * kChunkBytes;
  // KV-cache units hold one Q tile (both tiles read the same rows) and store
  // O row by row, so that room goes to a deeper K/V ring
  static constexpr int kQBufs = KVC ? 1 : 2;
  static constexpr int kStages = KVC ? (D == 128 ? 5 : 12) : (D == 128 ? 4 : 8);  // K/V ring depth
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kKVOff = kQBufs * kTileBytes;
  // plain: output staging for the TMA store of the epilogue, 128 rows x 64
  // columns (128B-swizzled) per query tile; KV cache: the row max / sum
  // exchange of the two tiles (2 x 2 x 128 floats)
  static constexpr uint32_t kStageOff = kKVOff + kStages * kTileBytes;
  static constexpr uint32_t kBarOff = kStageOff + (KVC ? 2048 : 2 * kChunkBytes);
  // barriers: q_full[2], q_empty[2], kv_full[S], kv_empty[S], s_full[2],
  //           p_half[2][2], o_ready[2], o_free[2], drain, v_fixed[S] (FIX)
  static constexpr int kNumBars = 4 + (FIX ? 3 : 2) * kStages + 11;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kBytes = kMiscOff + 16;
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

// Bounded wait like wait_bar, polling the phase without suspending the thread
// (MMA issuers waiting for P: a suspended thread wakes ~200 cycles after the
// phase completes, and the tensor pipe, whose MMA queue is about one
// instruction deep, idles for as long as the issuer is late).
__device__ __forceinline__ bool wait_bar_spin(uint32_t bar, uint32_t parity,
                                              volatile int *abort_flag, long long limit,
                                              int *status) {
  if (mbar_test_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
#pragma unroll
    for (int k = 0; k < 8; ++k)
      if (mbar_test_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) {
      record_status(status, 4);
      *abort_flag = 1;
      return false;
    }
  }
}

struct Work {
  int valid;
  int split;         // K/V split of the unit (0 without split-KV)
  int b, head[2], hkv;
  int m0[2];         // first query row of each tile within its sequence
  int lq, lk;        // sequence lengths
  int q_row0;        // tensor-map row of query row 0 of the sequence
  int k_row0;        // tensor-map row of key 0 of the sequence
  int map_b;         // tensor-map batch coordinate
  int64_t o_row0;    // global token index of query row 0 of the sequence
  int n_kv[2];       // K/V tiles each query tile visits ...
  int kv_begin[2];   // ... starting at this K/V tile of the sequence
  int kv_ub;         // first K/V tile loaded for the unit (min over its tiles)
  int n_max;         // K/V tiles loaded for the unit (the union of both ranges)
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

// K/V tiles visited by the query tile of rows [m0, m0 + 128) under a local
// window (kernels with score variants): keys [lo, hi] where lo is the left
// bound of the first row and hi the right bound of the last row.  Returns the
// count and sets *begin.  With both bounds >= 0 or unbounded, the ranges of two
// consecutive row tiles overlap or touch, so their union is contiguous.
__device__ __forceinline__ int window_kv_range(const FwdParams &p, int m0, int lq, int lk,
                                               int *begin, int rows = kBlockM) {
  *begin = 0;
  if (m0 >= lq || lk <= 0) return 0;
  const int off = lk - lq;
  const int last_row = min(m0 + rows, lq) - 1;
  const int lo = p.win_l < 0 ? 0 : max(0, m0 + off - p.win_l);
  const int hi = p.win_r < 0 ? lk - 1 : min(lk - 1, last_row + off + p.win_r);
  if (hi < lo) return 0;
  *begin = lo / kBlockN;
  return hi / kBlockN - *begin + 1;
}

// The i-th unit of this CTA (snake over the heavy-first unit order).
__device__ __forceinline__ int unit_of(int i) {
  const int G = gridDim.x;
  return i * G + ((i & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
}

// Decode work unit `unit`; every lane of the calling warp gets the same record.
// Dense: the row-unit index (heaviest causal rows first) is the slowest-varying
// part of the unit index.  Packed: units are numbered sequence by sequence
// (heaviest rows of a sequence first); the warp scans cu_seqlens cooperatively.
// Cut a unit's K/V tile range [*b, *b + *n) to split `split` of its sequence's
// nt tiles (chunks of ceil(nt / num_splits) tiles).
__device__ __forceinline__ void split_range(const FwdParams &p, int split, int lk, int *b,
                                            int *n) {
  const int nt = (lk + kBlockN - 1) / kBlockN;
  const int chunk = (nt + p.num_splits - 1) / p.num_splits;
  const int lo = split * chunk, hi = min(nt, lo + chunk);
  const int bb = max(*b, lo), e = min(*b + *n, hi);
  *n = max(0, e - bb);
  *b = bb;
}

// KV-cache unit: (split, K/V head, token block, sequence), split fastest.
__device__ inline Work decode_work_kvc(const FwdParams &p, int unit, int lane) {
  Work w;
  w.valid = 0;
  w.split = 0;
  if (p.num_splits > 1) {
    const int u = fast_div(p.div_splits, unit);
    w.split = unit - u * p.num_splits;
    unit = u;
  }
  const int u_h = fast_div(p.div_Hkv, unit);
  const int hkv = unit - u_h * p.Hkv;
  const int b = fast_div(p.div_tok_blocks, u_h);
  const int tb = u_h - b * p.tok_blocks;
  if (b >= p.B) return w;
  const int lk = p.cache_seqlens[b];
  const int64_t cap = p.block_table ? (int64_t)p.max_blocks * p.page_rows : p.page_rows;
  if (lk < 0 || lk > cap) {
    if (lane == 0) record_status(p.status, 5);
    return w;
  }
  w.b = b;
  w.hkv = hkv;
  w.head[0] = w.head[1] = hkv * p.group;
  w.lq = p.Sq;
  w.lk = lk;
  w.m0[0] = w.m0[1] = tb * p.tok_per_tile;
  w.q_row0 = 0;
  w.k_row0 = 0;
  w.map_b = b;
  w.o_row0 = (int64_t)b * p.Sq;
  int lo = 0;
  int n = window_kv_range(p, w.m0[0], w.lq, w.lk, &lo, p.tok_per_tile);
  if (p.num_splits > 1) split_range(p, w.split, lk, &lo, &n);
  // tile 0 reads K/V tiles lo, lo + 2, ...; tile 1 reads lo + 1, lo + 3, ...
  w.kv_ub = lo;
  w.n_max = n;
  w.kv_begin[0] = lo;
  w.kv_begin[1] = lo + 1;
  w.n_kv[0] = (n + 1) / 2;
  w.n_kv[1] = n / 2;
  w.valid = 1;
  return w;
}

// WIDE (head dim 256): one 128-row query tile per unit; tile 1 is left empty.
template <bool CAUSAL, bool VARLEN, bool EXT, bool WIDE = false>
__device__ Work decode_work(const FwdParams &p, int unit, int lane) {
  Work w;
  w.valid = 0;
  w.split = 0;
  if (EXT && p.num_splits > 1) {  // splits of one unit are adjacent: heavy units stay first
    const int u = fast_div(p.div_splits, unit);
    w.split = unit - u * p.num_splits;
    unit = u;
  }
  const int u_hu = fast_div(p.div_head_units, unit);  // unit / head_units
  int hu = unit - u_hu * p.head_units;
  int b = 0, ru = 0, n_ru = 0;
  if (!VARLEN) {
    n_ru = p.dense_row_units;
    if (p.rows_fastest) {
      // unit = (b * head_units + hu) * n_ru + ru
      const int bh = fast_div(p.div_ru, unit);
      ru = unit - bh * n_ru;
      b = fast_div(p.div_head_units, bh);
      hu = bh - b * p.head_units;
      if (b >= p.B) return w;
    } else {
      // unit = (ru * B + b) * head_units + hu: heavier rows first
      ru = fast_div(p.div_B, u_hu);
      b = u_hu - ru * p.B;
      if (ru >= n_ru) return w;
    }
    w.lq = p.Sq;
    w.lk = p.Sk;
    w.q_row0 = 0;
    w.k_row0 = 0;
    w.map_b = b;
    w.o_row0 = (int64_t)b * p.Sq;
  } else {
    const int idx = u_hu;
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
    if (found < 0) return w;
    b = found;
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1];
    const int k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    if (q0 < 0 || q1 < q0 || q1 > p.Sq || k0 < 0 || k1 < k0 || k1 > p.Sk) {
      if (lane == 0) record_status(p.status, 5);
      return w;
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
  if (CAUSAL || (EXT && p.reverse_rows)) ru = n_ru - 1 - ru;  // heavier (later) rows first
  w.b = b;
  if (WIDE) {
    w.head[0] = w.head[1] = hu;
    w.m0[0] = ru * kBlockM;
    w.m0[1] = w.lq;  // no rows
  } else if (p.pair_heads) {
    w.head[0] = 2 * hu;
    w.head[1] = 2 * hu + 1;
    w.m0[0] = w.m0[1] = ru * kBlockM;
  } else {
    w.head[0] = w.head[1] = hu;
    w.m0[0] = ru * 2 * kBlockM;
    w.m0[1] = ru * 2 * kBlockM + kBlockM;
  }
  w.hkv = w.head[0] / p.group;
  if (EXT) {
    w.n_kv[0] = window_kv_range(p, w.m0[0], w.lq, w.lk, &w.kv_begin[0]);
    w.n_kv[1] = window_kv_range(p, w.m0[1], w.lq, w.lk, &w.kv_begin[1]);
  } else {
    w.n_kv[0] = tile_kv_count<CAUSAL>(w.m0[0], w.lq, w.lk);
    w.n_kv[1] = tile_kv_count<CAUSAL>(w.m0[1], w.lq, w.lk);
    w.kv_begin[0] = w.kv_begin[1] = 0;
  }
  if (EXT && p.num_splits > 1) {
    // split s keeps K/V tiles [s c, s c + c) of the sequence, c = ceil(tiles / splits);
    // cutting two overlapping or touching ranges at the same bounds keeps
    // their union contiguous
    split_range(p, w.split, w.lk, &w.kv_begin[0], &w.n_kv[0]);
    split_range(p, w.split, w.lk, &w.kv_begin[1], &w.n_kv[1]);
  }
  if (w.n_kv[0] == 0 && w.n_kv[1] == 0) {
    w.kv_ub = 0;
    w.n_max = 0;
  } else {
    const int b0 = w.n_kv[0] ? w.kv_begin[0] : w.kv_begin[1];
    const int b1 = w.n_kv[1] ? w.kv_begin[1] : w.kv_begin[0];
    w.kv_ub = min(b0, b1);
    w.n_max = max(w.kv_begin[0] + w.n_kv[0], w.kv_begin[1] + w.n_kv[1]) - w.kv_ub;
  }
  w.valid = 1;
  return w;
}

// Keys of the unit's last K/V tile that belong to the sequence, when the tile
// reaches past the sequence's last key into memory that holds other data --
// the next packed sequence, or cache rows past the cached length -- and 0
// otherwise (dense problems: rows past the tensor read as zero).  Masked keys
// get P = 0, but 0 * Inf or 0 * NaN in O += P V would still be NaN, so those
// V rows are zeroed in shared memory before the tile is used.
template <bool VARLEN, bool KVC>
__device__ __forceinline__ int v_tail_rows(const Work &w) {
  if (!(VARLEN || KVC) || !w.valid || w.n_max == 0) return 0;
  const int valid = w.lk - (w.kv_ub + w.n_max - 1) * kBlockN;
  return valid < kBlockN ? valid : 0;
}

// Field of tile t of a Work record.  The tile index of a role is a run-time
// value; indexing the record's arrays with it would place the whole record in
// local memory (a round trip to L2 at every unit, since shared memory leaves
// little L1), so the field is selected instead.
__device__ __forceinline__ int tile_field(const int (&a)[2], int t) { return t ? a[1] : a[0]; }

// 16-bit pair of P values (low half = first key).
template <bool BF16>
__device__ __forceinline__ uint32_t pack_p(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

// Max of 32 scores (three-input max tree, depth 4).
__device__ __forceinline__ float max32(const float *x) {
  float a[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float *y = x + 8 * q;
    a[q] = fmax3(fmax3(y[0], y[1], y[2]), fmax3(y[3], y[4], y[5]), fmaxf(y[6], y[7]));
  }
  return fmax3(a[0], a[1], fmaxf(a[2], a[3]));
}

// P for 32 keys: exp2(s * scale_log2 - m * scale_log2) with the subtraction as
// packed FMAs, summed (fp32, before rounding) into four packed accumulators,
// rounded to 16-bit pairs and stored as 16 TMEM columns at `p_addr`.
template <bool BF16>
__device__ __forceinline__ void softmax_chunk(const float *x, float scale_log2, float ms,
                                              float2 (&acc)[4], uint32_t p_addr) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    float y0, y1;
    fma_f32x2(y0, y1, x[2 * i], x[2 * i + 1], scale_log2, scale_log2, -ms, -ms);
    const float p0 = ex2(y0), p1 = ex2(y1);
    add_f32x2(acc[i & 3].x, acc[i & 3].y, p0, p1);
    pk[i] = pack_p<BF16>(p0, p1);
  }
  tmem_st16(p_addr, pk);
}

// Score variants an instance with EXT carries code for (window bounds and
// split-KV always): a soft cap, ALiBi.  Each instance holds only the code of
// its own variants; the softmax's instruction stream stays short.
constexpr int kVarCap = 1;
constexpr int kVarAlibi = 2;

template <int D, bool BF16, bool CAUSAL, bool VARLEN, bool EXT, bool KVC = false,
          int VAR = kVarCap | kVarAlibi>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
  using L = Smem<D, KVC, VARLEN || KVC>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  auto q_full = [&](int t) { return bar0 + 8u * t; };
  auto q_empty = [&](int t) { return bar0 + 8u * (2 + t); };
  auto kv_full = [&](int s) { return bar0 + 8u * (4 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (4 + L::kStages + s); };
  auto s_full = [&](int t) { return bar0 + 8u * (4 + 2 * L::kStages + t); };
  // P_t of keys [64 h, 64 h + 64) is in tensor memory
  auto p_half = [&](int t, int h) { return bar0 + 8u * (6 + 2 * L::kStages + 2 * t + h); };
  auto o_ready = [&](int t) { return bar0 + 8u * (10 + 2 * L::kStages + t); };
  auto o_free = [&](int t) { return bar0 + 8u * (12 + 2 * L::kStages + t); };
  const uint32_t drain_bar = bar0 + 8u * (14 + 2 * L::kStages);
  // the V tile in ring slot s has had its rows past the sequence's keys zeroed
  auto v_fixed = [&](int s) { return bar0 + 8u * (15 + 2 * L::kStages + s); };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
  volatile int *mma_turn = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 8);
  // K/V loads the producer has issued: a role that may run ahead of the ring
  // (the free-running issuers of KV-cache units, the V-row fixer) waits on a
  // ring slot's barrier only once its load is issued, so it never waits a
  // whole lap ahead of the slot (an mbarrier parity wait cannot tell laps k
  // and k - 2 apart)
  volatile int *kv_issued = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 12);
  static_assert(L::kAlloc <= 227 * 1024, "shared memory budget");

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  FA_TRACE_AT(tid == 0, 2047);

  if (tid == 0) {
    *abort_flag = 0;
    for (int t = 0; t < 2; ++t) {
      mbar_init(q_full(t), 1);
      mbar_init(q_empty(t), KVC ? 2 : 1);  // KV cache: both tiles read Q buffer 0
      mbar_init(s_full(t), 1);
      mbar_init(p_half(t, 0), 4);  // one arrival per softmax warp
      mbar_init(p_half(t, 1), 4);
      mbar_init(o_ready(t), 1);
      mbar_init(o_free(t), 4);
    }
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 2);  // one release per query tile
      if (VARLEN || KVC) mbar_init(v_fixed(s), 1);
    }
    mbar_init(drain_bar, 2);      // one per MMA issuer
    *mma_turn = 0;
    *kv_issued = 0;
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
    tma_prefetch_desc(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long limit = p.wait_limit;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return wait_bar(bar, par, abort_flag, limit, p.status);
  };

  if (warp >= 8) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 96;" ::: "memory");
    if (warp == kTmaWarp) {
      // ---------------------------------------------------------- TMA producer
      const uint64_t pol_q = policy_evict_first();
      const uint64_t pol_kv = policy_evict_last();
      int issued = 0;                  // K/V loads issued (ring index, across units)
      int q_loads0 = 0, q_loads1 = 0;  // Q loads per tile buffer
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int unit = unit_of(i);
        if (unit >= p.total_units) break;
        const Work w = (KVC ? decode_work_kvc(p, unit, lane) : decode_work<CAUSAL, VARLEN, EXT>(p, unit, lane));
        if (!w.valid) continue;
        if (lane == 0) {
          auto load_q = [&](int t) {
            int &q_loads = t ? q_loads1 : q_loads0;
            if ((KVC ? w.n_max : tile_field(w.n_kv, t)) == 0 || !ok) return;
            // the previous unit's Q_t is free once its last S_t = Q_t K^T is done
            if (q_loads > 0 && !wait(q_empty(t), (q_loads - 1) & 1)) {
              ok = false;
              return;
            }
            mbar_arrive_expect_tx(q_full(t), L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_4d(sbase + L::kQOff + t * L::kTileBytes + c * kChunkBytes, &tm_q,
                          q_full(t), c * 64, tile_field(w.head, t),
                          w.q_row0 + tile_field(w.m0, t), w.map_b, pol_q);
            ++q_loads;
          };
          // one K or V tile of unit tile j (which: 0 K, 1 V) into the next ring slot
          auto issue = [&](int which, int j, int page) {
            const int idx = issued;
            const int s = idx % L::kStages;
            if (idx >= L::kStages && !wait(kv_empty(s), ((idx / L::kStages) + 1) & 1)) {
              ok = false;
              return;
            }
            int k_row = w.k_row0 + (w.kv_ub + j) * kBlockN, k_b = w.map_b;
            if (KVC) {
              k_row = ((w.kv_ub + j) * kBlockN) % p.page_rows;
              k_b = page;
            }
            FA_TRACE_AT(idx < 256, 1536 + idx);
            mbar_arrive_expect_tx(kv_full(s), L::kTileBytes);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_4d(sbase + L::kKVOff + s * L::kTileBytes + c * kChunkBytes,
                          which == 0 ? &tm_k : &tm_v, kv_full(s), c * 64, w.hkv, k_row, k_b,
                          pol_kv);
            issued = idx + 1;
            if (VARLEN || KVC) *kv_issued = issued;
          };
          if constexpr (KVC) {
            // K runs one tile ahead of V: K0, K1, V0, K2, V1, ..., K(n-1), V(n-2),
            // V(n-1), so a K slot is refilled as soon as its S = Q K^T is done
            auto page_of = [&](int j) {
              int pg = w.map_b;
              if (p.block_table) {
                pg = __ldg(p.block_table + (int64_t)w.b * p.max_blocks +
                           ((w.kv_ub + j) * kBlockN) / p.page_rows);
                if (pg < 0 || pg >= p.num_pages) {
                  record_status(p.status, 5);
                  pg = 0;
                }
              }
              return pg;
            };
            load_q(0);  // one Q tile serves both
            int pg_cur = w.n_max > 0 ? page_of(0) : 0;
            if (w.n_max > 0 && ok) issue(0, 0, pg_cur);
            for (int j = 0; j < w.n_max && ok; ++j) {
              int pg_next = pg_cur;
              if (j + 1 < w.n_max) {
                pg_next = page_of(j + 1);
                issue(0, j + 1, pg_next);
              }
              if (ok) issue(1, j, pg_cur);
              pg_cur = pg_next;
            }
          } else {
            // Q0, K0, Q1, V0, K1, V1, ...: tile 0's first S needs only Q0 and
            // K0, and K0 does not wait behind the previous unit's last S1
            load_q(0);
            if (w.n_max > 0 && ok) issue(0, 0, 0);
            load_q(1);
            for (int j = 0; j < w.n_max && ok; ++j) {
              if (j > 0) issue(0, j, 0);
              if (ok) issue(1, j, 0);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (!ok && lane == 0) {
        // drain copies still in flight into the ring before the CTA exits
        for (int idx = max(0, issued - L::kStages); idx < issued; ++idx)
          wait_bar(kv_full(idx % L::kStages), (idx / L::kStages) & 1, abort_flag, limit,
                   p.status, false);
        if (q_loads0 > 0)
          wait_bar(q_full(0), (q_loads0 - 1) & 1, abort_flag, limit, p.status, false);
        if (q_loads1 > 0)
          wait_bar(q_full(1), (q_loads1 - 1) & 1, abort_flag, limit, p.status, false);
      }
    } else if ((warp == kMmaWarp || warp == kMmaWarp2)) {
      // ------------------------------------------------ MMA issuers, one per tile
      // Warp 8 lane 0 issues tile 0's MMAs, warp 10 lane 0 tile 1's.  A turn
      // flag in shared memory makes them take strict turns, bracket by bracket:
      //   [S0 = Q0 K(0)^T] [S1 = Q1 K(0)^T] [O0 += P0 V(0), S0 = Q0 K(1)^T]
      //   [O1 += P1 V(0), S1 = Q1 K(1)^T] ...
      // so the tensor pipe still alternates tiles (tile 0's softmax runs while
      // the pipe works on tile 1), while each issuer does its barrier waits and
      // commits during the other one's bracket: issue blocks on a shallow queue,
      // and one thread doing both left the pipe idle between brackets.
      const int T = (warp == kMmaWarp) ? 0 : 1;
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, kBlockM, D, true);
      // descriptors built once; each MMA adds a compile-time offset
      const uint64_t q_desc =
          make_sdesc_sw128(sbase + L::kQOff + (KVC ? 0 : T) * L::kTileBytes, 16, 1024);
      const uint64_t kv_desc0 = make_sdesc_sw128(sbase + L::kKVOff, 16, 1024);
      const uint64_t v_desc0 = make_sdesc_sw128(sbase + L::kKVOff, kChunkBytes, 1024);
      const uint32_t d_s = tmem + T * 128, d_o = tmem + 256 + T * D;
      auto issue_qk = [&](int kidx) {
        const uint64_t kd = kv_desc0 + (((kidx % L::kStages) * L::kTileBytes) >> 4);
        mma_ss(d_s, q_desc, kd, idesc_qk, 0u);
#pragma unroll
        for (int kk = 1; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss_acc(d_s, q_desc + off, kd + off, idesc_qk);
        }
      };
      // O_T += P_T V for keys [64 h, 64 h + 64): four K = 16 steps reading
      // P from TMEM columns [32 h, 32 h + 32) of S_T
      auto issue_pv_half = [&](int vidx, int h, bool first) {
        const uint64_t vd = v_desc0 + (((vidx % L::kStages) * L::kTileBytes + h * 4 * 2048) >> 4);
        const uint32_t a = d_s + h * 32;
        if (h == 0)
          mma_ts(d_o, a, vd, idesc_pv, first ? 0u : 1u);
        else
          mma_ts_acc(d_o, a, vd, idesc_pv);
#pragma unroll
        for (int kk = 1; kk < 4; ++kk)
          mma_ts_acc(d_o, a + kk * 8, vd + ((kk * 2048) >> 4), idesc_pv);
      };
      auto kv_par = [&](int idx) { return (uint32_t)((idx / L::kStages) & 1); };
      // bounded spin until the producer has issued ring load idx (KV cache)
      auto issued_past = [&](int idx) {
        if (*kv_issued > idx) return true;
        const long long t0 = clock64();
        while (*kv_issued <= idx) {
          if (*abort_flag) return false;
          if (clock64() - t0 > limit) {
            record_status(p.status, 4);
            *abort_flag = 1;
            return false;
          }
        }
        return true;
      };
      // bounded spin for this issuer's turn (the other one is issuing); the
      // flag is polled several times per abort / time-limit check, because
      // the tensor pipe runs dry while this thread waits to see it
      auto take_turn = [&]() {
        if (*mma_turn == T) return true;
        const long long t0 = clock64();
        while (true) {
#pragma unroll
          for (int k = 0; k < 8; ++k)
            if (*mma_turn == T) return true;
          if (*abort_flag) return false;
          if (clock64() - t0 > limit) {
            record_status(p.status, 4);
            *abort_flag = 1;
            return false;
          }
        }
      };
      auto pass_turn = [&]() { *mma_turn = 1 - T; };
      // P of the tile is polled (see wait_bar_spin)
      auto wait_p = [&](int h, uint32_t par) {
        return wait_bar_spin(p_half(T, h), par, abort_flag, limit, p.status);
      };
      // every K/V load is released by two arrivals, one per tile; a load the
      // other tile never reads gets both of them from this issuer
      auto release = [&](int idx, bool other_reads) {
        tc_commit(kv_empty(idx % L::kStages));
        if (!other_reads) mbar_arrive(kv_empty(idx % L::kStages));
      };
      int used = 0;    // K/V loads consumed (ring index, across units)
      int q_used = 0;  // Q tiles consumed
      int p_seen = 0;  // P tiles consumed (p_half phases)
      int o_done = 0;  // finished O accumulations (o_ready / o_free phases)
      uint32_t vpar = 0;  // bit s: phase parity of v_fixed(s)
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int unit = unit_of(i);
        if (unit >= p.total_units) break;
        const Work w = (KVC ? decode_work_kvc(p, unit, lane) : decode_work<CAUSAL, VARLEN, EXT>(p, unit, lane));
        if (!w.valid || w.n_max == 0) continue;
        // the unit's last load is a V tile whose rows past the sequence's keys
        // are zeroed by the fixer warp: whoever reads it also waits for that
        // (each issuer tracks every fix's phase, read or not)
        const bool vfix = v_tail_rows<VARLEN, KVC>(w) > 0;
        const int fix_idx = vfix ? used + 2 * w.n_max - 1 : -1;
        const int fix_slot = vfix ? fix_idx % L::kStages : 0;
        const uint32_t fix_par = (vpar >> fix_slot) & 1u;
        if (vfix) vpar ^= 1u << fix_slot;
        if (lane == 0 && KVC) {
          // KV-cache units: each tile owns every other load and the tensor
          // pipe is far from busy, so the issuers run free (no turns), and
          // O += P V of a tile's previous load is issued and its V slot
          // released before waiting for the next K: the producer refills the
          // ring without waiting for a K load to land first
          const int n = tile_field(w.n_kv, T), nm = w.n_max;
          const int off = tile_field(w.kv_begin, T) - w.kv_ub;
          // ring positions of the unit's loads (the producer's K-ahead order)
          auto kpos = [&](int u) { return u == 0 ? 0 : 2 * u - 1; };
          auto vpos = [&](int u) { return u + 1 < nm ? 2 * u + 2 : 2 * nm - 1; };
          if (nm > 0 && n == 0) {
            // reads no Q this unit: release it, but only once it has landed,
            // so the arrival cannot count towards the previous unit's phase
            ok = wait(q_full(0), q_used & 1);
            if (ok) mbar_arrive(q_empty(0));
          }
          for (int jq = 0; jq <= n && ok; ++jq) {
            const int u = off + 2 * jq;
            const int kidx = used + kpos(u), vidx = used + vpos(u - 2);
            if (jq >= 1) {
              ok = issued_past(vidx) && wait(kv_full(vidx % L::kStages), kv_par(vidx)) &&
                   (vidx != fix_idx || wait(v_fixed(fix_slot), fix_par)) &&
                   (jq > 1 || o_done == 0 || wait(o_free(T), (o_done - 1) & 1)) &&
                   wait_p(0, p_seen & 1);
              if (!ok) break;
              tc_fence_after();
              issue_pv_half(vidx, 0, jq == 1);
              if (!wait_p(1, p_seen & 1)) {
                ok = false;
                break;
              }
              ++p_seen;
              tc_fence_after();
              issue_pv_half(vidx, 1, false);
              if (jq == n) {
                tc_commit(o_ready(T));
                ++o_done;
              }
              release(vidx, false);
            }
            if (jq < n) {
              if (jq == 0) ok = wait(q_full(0), q_used & 1);
              ok = ok && issued_past(kidx) && wait(kv_full(kidx % L::kStages), kv_par(kidx));
              if (!ok) break;
              tc_fence_after();
              issue_qk(kidx);
              tc_commit(s_full(T));
              if (jq == n - 1) tc_commit(q_empty(0));
              release(kidx, false);
            }
          }
          if (nm > 0) ++q_used;  // one Q load per unit with keys
          used += 2 * w.n_max;
        } else if (!KVC && lane == 0) {
          const int n = tile_field(w.n_kv, T), n_other = tile_field(w.n_kv, 1 - T);
          // bracket u = 0 .. n_max of the unit: O_T += P_T V(u-1) if this
          // tile read load u-1, then S_T = Q_T K(u)^T if it reads load u.
          // Both issuers walk every bracket, so the turns stay paired even
          // when the tiles' K/V ranges differ (local windows).
          const int off = tile_field(w.kv_begin, T) - w.kv_ub;
          const int off_other = tile_field(w.kv_begin, 1 - T) - w.kv_ub;
          auto other_reads = [&](int u) {
            const int d = u - off_other;
            return d >= 0 && d < n_other;
          };
          for (int u = 0; u <= w.n_max && ok; ++u) {
            const int jq = u - off;  // this tile's step: S_T = Q_T K(jq)^T
            const bool qk = jq >= 0 && jq < n, pv = jq >= 1 && jq <= n;
            const int kidx = used + 2 * u, vidx = used + 2 * (u - 1) + 1;
            if (qk && jq == 0) {  // first S_T of the unit: Q_T must have landed
              ok = wait(q_full(T), q_used & 1);
              ++q_used;
            }
            // K/V (and, for a unit's first O += P V, the previous unit's
            // epilogue having read O_T out) are checked first: these barriers
            // completed long ago, and each check costs a shared-memory round
            // trip that now hides behind the wait for this tile's softmax
            if (ok && pv)
              ok = wait(kv_full(vidx % L::kStages), kv_par(vidx)) &&
                   (vidx != fix_idx || wait(v_fixed(fix_slot), fix_par)) &&
                   (jq > 1 || o_done == 0 || wait(o_free(T), (o_done - 1) & 1));
            if (ok && qk) ok = wait(kv_full(kidx % L::kStages), kv_par(kidx));
            if (ok && pv) ok = wait_p(0, p_seen & 1);
            FA_TRACE_AT(i == 0 && u < 64, 1024 + u * 8 + 2 + 2 * T);
            ok = ok && take_turn();
            if (!ok) break;
            tc_fence_after();
            if (pv) {
              // keys 0-63 go to the tensor pipe while the softmax still works
              // on keys 64-127; the turn is held until the bracket is complete
              issue_pv_half(vidx, 0, jq == 1);
              if (!wait_p(1, p_seen & 1)) {
                ok = false;
                break;
              }
              ++p_seen;
              tc_fence_after();
              issue_pv_half(vidx, 1, false);
            }
            if (qk) issue_qk(kidx);
            pass_turn();
            FA_TRACE_AT(i == 0 && u < 64, 1024 + u * 8 + 3 + 2 * T);
            if (pv) {
              if (jq == n) {
                tc_commit(o_ready(T));  // tile T of this unit is complete
                ++o_done;
              }
              release(vidx, other_reads(u - 1));
            }
            if (qk) {
              tc_commit(s_full(T));
              if (jq == n - 1) tc_commit(q_empty(T));  // last S_T of this unit issued
              release(kidx, other_reads(u));
            }
          }
          used += 2 * w.n_max;
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      if (lane == 0) {
        // make sure no MMA is still running when tensor memory is released
        tc_commit(drain_bar);
        wait_bar(drain_bar, 0, abort_flag, limit, p.status, false);
      }
    } else if (warp == kFixWarp && (VARLEN || KVC)) {
      // ------------------------------------------------- V rows past the keys
      // For each unit whose last K/V tile reaches past the sequence's keys:
      // once that V tile has landed, zero its rows past the last key (whole
      // 128-byte rows of each 64-column chunk, so the swizzle does not
      // matter), make the writes visible to the tensor core's proxy and
      // signal v_fixed of the slot.  The issuers hold the slot until then.
      int used = 0;
      bool ok = true;
      for (int i = 0; ok; ++i) {
        const int unit = unit_of(i);
        if (unit >= p.total_units) break;
        const Work w = (KVC ? decode_work_kvc(p, unit, lane) : decode_work<CAUSAL, VARLEN, EXT>(p, unit, lane));
        if (!w.valid || w.n_max == 0) continue;
        const int valid = v_tail_rows<VARLEN, KVC>(w);
        if (valid > 0) {
          const int idx = used + 2 * w.n_max - 1;  // ring index of the unit's last V load
          const int s = idx % L::kStages;
          // wait for the producer to issue the load (never a lap ahead of the
          // slot), then for the load itself
          const long long t0 = clock64();
          while (ok && *kv_issued <= idx) {
            __nanosleep(256);  // far ahead of the load: sleep, keep issue slots free
            if (*abort_flag) ok = false;
            if (clock64() - t0 > limit) {
              record_status(p.status, 4);
              *abort_flag = 1;
              ok = false;
            }
          }
          ok = __all_sync(0xffffffffu, ok && wait(kv_full(s), (idx / L::kStages) & 1));
          if (ok) {
            const uint32_t tile = sbase + L::kKVOff + s * L::kTileBytes;
#pragma unroll 1
            for (int c = 0; c < L::kChunks; ++c)
#pragma unroll 1
              for (uint32_t b = (uint32_t)valid * 128u + lane * 16u; b < kChunkBytes; b += 512u)
                st_shared_v4(tile + c * kChunkBytes + b, 0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(v_fixed(s));
          }
        }
        used += 2 * w.n_max;
      }
    }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 192;" ::: "memory");
    // ------------------------------------------------------ softmax + epilogue
    const int t = warp >> 2;        // query tile of this warpgroup
    const int quarter = warp & 3;   // TMEM lane quarter
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t s_addr = lane_base + t * 128;
    const uint32_t o_addr = lane_base + 256 + t * D;
    // raw scores (plain kernels, and local windows alone) fold scale * log2(e)
    // into the exps; a soft cap or ALiBi turns every score into log2 units
    // first, and so does the KV-cache path, whose two-tile merge works in log2
    // units
    // the variants this instance carries code for (the others are off)
    const float cap_k = (VAR & kVarCap) ? p.cap_k : 0.f;
    const float *const alibi = (VAR & kVarAlibi) ? p.alibi : nullptr;
    const bool raw_scores = !EXT || (!KVC && cap_k == 0.f && alibi == nullptr);
    // a soft cap alone keeps tanh(scale s / c) as the score and folds its
    // factor c log2(e) into the exps, as the plain path folds scale log2(e)
    const bool cap_folded = EXT && !KVC && cap_k != 0.f && alibi == nullptr;
    const float scale_log2 = raw_scores ? p.scale_log2 : (cap_folded ? p.cap_l2 : 1.f);
    const float neg_thr = -p.threshold;
    // every lane of a warp must agree before the warp-wide tcgen05.ld / st
    auto warp_wait = [&](uint32_t bar, uint32_t parity) {
      const bool got = wait(bar, parity);
      return __all_sync(0xffffffffu, got);
    };
    int s_seen = 0;   // S tiles consumed (s_full phases, across units)
    int o_seen = 0;   // finished units of this tile (o_ready phases)
    [[maybe_unused]] int x_units = 0;  // KV-cache units merged (exchange buffer parity)
    const bool elected = quarter == 0 && lane == 0;  // issues this tile's TMA stores
    const uint32_t stage = sbase + L::kStageOff + t * kChunkBytes;
    // The warpgroup meets at named barrier 1 + t in the epilogue.  To keep every
    // barrier complete, the role never leaves its unit loop early: after a
    // failed wait (ok == false) it keeps walking the same units and barriers
    // but skips every wait, tensor-memory access and store.
    bool ok = true;
    for (int i = 0;; ++i) {
      const int unit = unit_of(i);
      if (unit >= p.total_units) break;
      const Work w = (KVC ? decode_work_kvc(p, unit, lane) : decode_work<CAUSAL, VARLEN, EXT>(p, unit, lane));
      if (!w.valid || tile_field(w.m0, t) >= w.lq) continue;  // no rows of this tile
      const int m0 = tile_field(w.m0, t);  // per-tile fields read once per unit
      const int n_kv = tile_field(w.n_kv, t);
      const int lq = w.lq, lk = w.lk;
      // query row within its sequence and its head (KV-cache tiles pack
      // (token, head) pairs: row r is token m0 + r / group, head r % group)
      const int qi = KVC ? m0 + row / p.group : m0 + row;
      const int head_t = tile_field(w.head, t);
      const int head = KVC ? head_t + row % p.group : head_t;
      const int diag = qi + lk - lq;  // last visible key of this row (causal)
      [[maybe_unused]] const int kv_begin = tile_field(w.kv_begin, t);
      [[maybe_unused]] const float slope_l2 =
          (EXT && alibi) ? alibi[head] * 1.4426950408889634f : 0.f;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < n_kv && ok; ++j) {
        if (!warp_wait(s_full(t), s_seen & 1)) { ok = false; break; }
        ++s_seen;
        [[maybe_unused]] const bool tr = i == 0 && quarter == 0 && lane == 0 && j < 63;
        FA_TRACE_AT(tr, (t * 64 + j) * 8);
        tc_fence_after();
        uint32_t sr[128];
        tmem_ld128_wait(s_addr, sr);
        float *s = reinterpret_cast<float *>(sr);
        FA_TRACE_AT(tr, (t * 64 + j) * 8 + 1);
        const int k0 = (EXT ? kv_begin + (KVC ? 2 * j : j) : j) * kBlockN;
        if constexpr (EXT) {
          // scores in log2 units: soft cap c tanh(scale s / c) with the
          // hardware tanh, then the ALiBi penalty -slope |diag - key|
          const int last_row = min(m0 + (KVC ? p.tok_per_tile : kBlockM), lq) - 1;
          if (cap_folded) {
            soft_cap<kBlockN, false>(s, cap_k, 1.f);
          } else if (cap_k != 0.f) {
            soft_cap<kBlockN, true>(s, cap_k, p.cap_l2);
          } else if (!raw_scores && !alibi) {
            const float sl2 = p.scale_log2;
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) s[c] *= sl2;
          }
          if (alibi) {
            // after the soft cap the scores are in log2 units already
            const float mul = cap_k != 0.f ? 1.f : p.scale_log2;
            const float d0 = (float)(diag - k0);
            const int first_diag = m0 + lk - lq, last_diag = last_row + lk - lq;
            if (k0 + kBlockN - 1 <= first_diag || k0 >= last_diag) {
              // the whole tile lies on one side of every row's diagonal, where
              // -slope |d0 - c| = sg (c - d0) is linear in the key: two packed
              // FMAs per key pair
              const float sg = k0 >= last_diag ? -slope_l2 : slope_l2;
              const float base = -sg * d0;
#pragma unroll
              for (int c = 0; c < kBlockN; c += 2) {
                float b0, b1;
                fma_f32x2(b0, b1, sg, sg, (float)c, (float)(c + 1), base, base);
                fma_f32x2(s[c], s[c + 1], s[c], s[c + 1], mul, mul, b0, b1);
              }
            } else {
#pragma unroll
              for (int c = 0; c < kBlockN; ++c)
                s[c] = fmaf(-slope_l2, fabsf(d0 - (float)c), s[c] * mul);
            }
          }
          const bool need_mask = (k0 + kBlockN > lk) ||
                                 (p.win_r >= 0 && k0 + kBlockN - 1 > m0 + lk - lq + p.win_r) ||
                                 (p.win_l >= 0 && k0 < last_row + lk - lq - p.win_l);
          if (need_mask) {
            // keys [lo, hi) of this tile are visible to the row; a warp none
            // of whose rows has its left bound inside the tile (causal, or a
            // right bound alone) takes the one-sided select
            const int lo = p.win_l < 0 ? 0 : diag - p.win_l - k0;
            const int hi = min(lk, p.win_r < 0 ? lk : diag + p.win_r + 1) - k0;
            if (__all_sync(0xffffffffu, lo <= 0)) {
#pragma unroll
              for (int c = 0; c < kBlockN; ++c) s[c] = (c < hi) ? s[c] : -INFINITY;
            } else {
#pragma unroll
              for (int c = 0; c < kBlockN; ++c) s[c] = (c >= lo && c < hi) ? s[c] : -INFINITY;
            }
          }
        } else if ((k0 + kBlockN > lk) || (CAUSAL && (k0 + kBlockN - 1 > m0 + lk - lq))) {
          int lim = lk - k0;  // keys [0, lim) of this tile are visible to the row
          if (CAUSAL) lim = min(lim, diag - k0 + 1);
#pragma unroll
          for (int c = 0; c < kBlockN; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
        }
        const float bm = fmax3(fmaxf(max32(s), max32(s + 32)), max32(s + 64), max32(s + 96));
        float alpha = 1.f;
        bool rescale = false;
        if (j == 0) {
          m = bm;  // the first tile sets the max, no threshold
        } else {
          const float m_cur = fmaxf(m, bm);
          const float diff = (m_cur == -INFINITY) ? 0.f : (m - m_cur) * scale_log2;
          if (!(diff >= neg_thr)) {  // rise above the threshold: rescale
            alpha = ex2(diff);
            m = m_cur;
            rescale = true;
          }                          // else skip and keep the lagged max
        }
        FA_TRACE_AT(tr, (t * 64 + j) * 8 + 2);
        if (__any_sync(0xffffffffu, rescale)) {
          // O_t holds P V up to tile j-1: S_t(j) was committed after that PV,
          // so it has completed and no MMA writes O_t until this P is ready
          l *= alpha;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32_wait(o_addr + c * 32, orr);
#pragma unroll
            for (int k = 0; k < 32; ++k)
              orr[k] = __float_as_uint(__uint_as_float(orr[k]) * alpha);
            tmem_st32(o_addr + c * 32, orr);
          }
        }
        const float ms = (m == -INFINITY) ? 0.f : m * scale_log2;
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                         make_float2(0.f, 0.f)};
        // P of keys 0-63 is handed over before keys 64-127 are computed, so
        // O += P V for the first half overlaps the second half's exps
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          softmax_chunk<BF16>(s + 32 * c, scale_log2, ms, acc, s_addr + 16 * c);
          if (c & 1) {
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(p_half(t, c >> 1));
            FA_TRACE_AT(tr, (t * 64 + j) * 8 + 3 + (c >> 1));
          }
        }
        add_f32x2(acc[0].x, acc[0].y, acc[1].x, acc[1].y);
        add_f32x2(acc[2].x, acc[2].y, acc[3].x, acc[3].y);
        add_f32x2(acc[0].x, acc[0].y, acc[2].x, acc[2].y);
        l += acc[0].x + acc[0].y;
      }
      // ------------------------------------------------------------- epilogue
      [[maybe_unused]] const bool tr = i == 0 && quarter == 0 && lane == 0;
      FA_TRACE_AT(tr, (t * 64 + 63) * 8 + 5);
      // The fields only the epilogue needs (sequence, output row base, tensor
      // map coordinates, split) are decoded again here from an opaque copy of
      // the unit counter, so they hold no registers through the K/V loop.
      int i_e;
      asm volatile("mov.b32 %0, %1;" : "=r"(i_e) : "r"(i));
      const int unit_e = unit_of(i_e);
      const Work we = KVC ? decode_work_kvc(p, unit_e, lane)
                          : decode_work<CAUSAL, VARLEN, EXT>(p, unit_e, lane);
      // O_t of this unit (zero when no key is visible), read out of tensor
      // memory and released first so the next unit's O += P V can start
      uint32_t orr[D];
#pragma unroll
      for (int k = 0; k < D; ++k) orr[k] = 0u;
      if constexpr (KVC) {
        // both tiles hold the same rows over even / odd K/V tiles: tile 1
        // hands its row max and sum to tile 0 through shared memory
        // (double-buffered by unit), tile 0 reads
        // both accumulators out of tensor memory and merges them:
        //   M = max(m0, m1), O = O0 2^(m0 - M) + O1 2^(m1 - M), l likewise
        float *xm = reinterpret_cast<float *>(smem + L::kStageOff) + (x_units & 1) * 256;
        float *xl = xm + 128;
        ++x_units;
        if (n_kv > 0 && ok) {
          ok = warp_wait(o_ready(t), o_seen & 1);
          ++o_seen;
        }
        if (t == 1) {
          xm[row] = (l > 0.f && ok) ? m : -INFINITY;
          xl[row] = ok ? l : 0.f;
          tc_fence_before();
          named_barrier_sync(3, 256);
          continue;  // tile 0 stores the merged rows
        }
        named_barrier_sync(3, 256);
        tc_fence_after();
        const int n1 = we.n_kv[1];
        const float m1 = xm[row], l1 = xl[row];
        const float mine = l > 0.f ? m : -INFINITY;
        const float mx = fmaxf(mine, m1);
        const float a0 = mine == -INFINITY ? 0.f : ex2(mine - mx);
        const float a1 = m1 == -INFINITY ? 0.f : ex2(m1 - mx);
        if (ok) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o1[32];
            if (n_kv > 0) tmem_ld32_wait(o_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(orr + 32 * c));
            if (n1 > 0) {
              tmem_ld32_wait(o_addr + D + c * 32, o1);
#pragma unroll
              for (int k = 0; k < 32; ++k)
                orr[32 * c + k] = __float_as_uint(__uint_as_float(orr[32 * c + k]) * a0 +
                                                  __uint_as_float(o1[k]) * a1);
            } else {
#pragma unroll
              for (int k = 0; k < 32; ++k)
                orr[32 * c + k] = __float_as_uint(__uint_as_float(orr[32 * c + k]) * a0);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if (n_kv > 0) mbar_arrive(o_free(0));
            if (n1 > 0) mbar_arrive(o_free(1));
          }
        }
        l = l * a0 + l1 * a1;
        m = mx;
      } else if (n_kv > 0 && ok) {
        ok = warp_wait(o_ready(t), o_seen & 1);
        ++o_seen;
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
            tmem_ld32(o_addr + c * 32, *reinterpret_cast<uint32_t(*)[32]>(orr + 32 * c));
#pragma unroll
          for (int c = 0; c < D / 32; ++c)
            tmem_wait_ld32(*reinterpret_cast<uint32_t(*)[32]>(orr + 32 * c));
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(o_free(t));
        }
      }
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool row_valid = qi < lq;
      const int64_t tok = we.o_row0 + qi;
      auto packed = [&](int k) {  // 16-bit pair of normalised O columns 2k, 2k+1
        return pack_p<BF16>(__uint_as_float(orr[2 * k]) * inv_l,
                            __uint_as_float(orr[2 * k + 1]) * inv_l);
      };
      const int64_t li = VARLEN ? (int64_t)head * p.Sq + tok
                                : ((int64_t)we.b * p.Hq + head) * p.Sq + qi;
      const float lse = (l > 0.f) ? (m * scale_log2 + log2f(l)) * 0.69314718055994531f
                                  : -INFINITY;
      // a packed tile cut by its sequence end would spill into the next
      // sequence through the tensor map, so it is stored row by row instead
      const bool use_tma = !KVC && (!VARLEN || (m0 + kBlockM <= lq));
      if (EXT && p.num_splits > 1) {
        // split-KV partial: normalised fp32 O_s and LSE_s of this split
        if (row_valid && ok) {
          const int64_t slot = (int64_t)we.split * p.part_rows + li;
          float4 *dst = reinterpret_cast<float4 *>(p.o_part + slot * D);
#pragma unroll
          for (int k = 0; k < D / 4; ++k)
            dst[k] = make_float4(__uint_as_float(orr[4 * k]) * inv_l,
                                 __uint_as_float(orr[4 * k + 1]) * inv_l,
                                 __uint_as_float(orr[4 * k + 2]) * inv_l,
                                 __uint_as_float(orr[4 * k + 3]) * inv_l);
          p.lse_part[slot] = lse;
        }
      } else if (use_tma) {
        // O leaves in 32-column quarters through the two 8 KB halves of the
        // tile's staging buffer, quarter q through half q % 2.  Before the
        // warpgroup meets after writing a quarter, the elected thread waits
        // until the store from the other half has read it, so the next
        // quarter can be written there while this one is being read; the
        // last store of a unit is only waited for when its half is next
        // written.
#pragma unroll
        for (int qd = 0; qd < D / 32; ++qd) {
          const uint32_t buf = stage + (qd & 1) * (kChunkBytes / 2);
          if (ok) {
            // row `row`, 16-byte chunk c at swizzled position c ^ ((row / 2) % 4)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int k = qd * 16 + 4 * c;
              st_shared_v4(buf + row * 64 + ((c ^ ((row >> 1) & 3)) << 4), packed(k),
                           packed(k + 1), packed(k + 2), packed(k + 3));
            }
            fence_proxy_async_smem();
          }
          if (elected) bulk_wait_group_read0();  // the other half is free again
          named_barrier_sync(1 + t, 128);
          if (elected && ok) {
            tma_store_4d(&tm_o, buf, qd * 32, tile_field(we.head, t), we.q_row0 + m0, we.map_b);
            bulk_commit_group();
          }
        }
      } else if (row_valid && ok) {
        elem_t *o = reinterpret_cast<elem_t *>(p.o) + (tok * p.Hq + head) * (int64_t)D;
        uint4 *dst = reinterpret_cast<uint4 *>(o);
#pragma unroll
        for (int k = 0; k < D / 8; ++k)
          dst[k] = make_uint4(packed(4 * k), packed(4 * k + 1), packed(4 * k + 2), packed(4 * k + 3));
      }
      if (row_valid && ok && p.lse != nullptr && !(EXT && p.num_splits > 1)) p.lse[li] = lse;
      FA_TRACE_AT(tr, (t * 64 + 63) * 8 + 6);
    }
    if (elected) bulk_wait_group0();  // output stores complete before the CTA exits
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
