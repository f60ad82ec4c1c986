// Backward pass of exact attention on sm_103a (see fa_bwd.cuh for the math).
//
// Both tile passes use the same two tcgen05 patterns as the forward kernel:
//   SS, both operands K-major, K = D:  S^T = K Q^T, dP^T = V dO^T (key pass,
//                                      M128 N64 per half of the queries),
//                                      S = Q K^T, dP = dO V^T (query pass,
//                                      M128 N128);
//   TS, A = 16-bit P / dS in tensor memory, B MN-major, M128 N=D, K = 64
//                                      rows per half: dV += P^T dO,
//                                      dK += dS^T Q (key pass), dQ += dS K
//                                      (query pass).
// Both tile passes are persistent: one CTA per SM walks a snake over the
// heavy-first order of its work items, every barrier phase carried across
// items.
// A CTA has ten warps: warps 0-7 do the elementwise work (warp w owns tensor
// memory lanes 32 (w % 4) .. 32 (w % 4) + 31 -- one key row per thread in the
// key pass, one query row in the query pass -- and warpgroup w / 4 the column
// half 64 (w / 4) .. 64 (w / 4) + 63, so two warps share each sub-partition),
// warp 8 issues the TMA loads, warp 9 owns the tensor memory and issues the
// MMAs (one elected lane).  Per tile step the MMA pair
// that produces the scores and dP runs, the elementwise warps turn them into
// P / dS (16-bit, written over the scores in tensor memory), and the MMAs
// that consume them run; the tensor pipe executes one thread's MMAs in issue
// order, so the next step's score MMA cannot overwrite P before it is read.
// Every wait is bounded (timeout -> FA_ERR_TIMEOUT in the status word); after
// a failed wait a role keeps walking its loop without waiting, so every named
// barrier still completes, and in-flight copies and MMAs are drained before
// shared and tensor memory are released.
#include "fa_bwd.cuh"
#include "fa_launch.cuh"

namespace fa {
namespace {

constexpr int kBwdThreads = 320;
constexpr int kBwdProducer = 8;
constexpr int kBwdMma = 9;

template <int D>
struct SmemBwd {
  static constexpr uint32_t kTile = (D / 64) * kChunkBytes;  // 128 rows x D, 16-bit
  // resident pair (key pass: K, V; query pass: Q, dO) and two stages of the
  // streamed pair (key pass: Q, dO; query pass: K, V)
  static constexpr uint32_t kResOff = 0;
  static constexpr uint32_t kStOff = 2 * kTile;
  static constexpr uint32_t kVecOff = kStOff + 4 * kTile;  // [2][2][128] floats (key pass)
  static constexpr uint32_t kBarOff = kVecOff + 2048;
  static constexpr int kNumBars = 15;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  // key pass: a 2 KB staging buffer per elementwise warp for the dV / dK rows
  static constexpr uint32_t kEpiOff = (kMiscOff + 16 + 127) / 128 * 128;
  static constexpr uint32_t kBytes = kEpiOff + 8 * 2048;
  // at least 120 KB, so that two CTAs never share an SM: each allocates all
  // 512 tensor-memory columns
  static constexpr uint32_t kAlloc = kBytes + 1024 > 120u * 1024 ? kBytes + 1024 : 120u * 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// Dynamic shared memory opt-in, once per device and library epoch.
struct BwdOptIn {
  std::atomic<unsigned long long> bits{0};
  std::atomic<unsigned> epoch{0};
  template <class Kernel>
  cudaError_t ensure(Kernel kern, int bytes, int device) {
    const unsigned ep = launch_epoch().load(std::memory_order_acquire);
    if (epoch.load(std::memory_order_acquire) != ep) {
      bits.store(0, std::memory_order_release);
      epoch.store(ep, std::memory_order_release);
    }
    const unsigned long long bit = 1ull << (device & 63);
    if (bits.load(std::memory_order_acquire) & bit) return cudaSuccess;
    const cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) bits.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  }
};

// ---------------------------------------------------------------- row pass
// Delta = rowsum(dO * O) in fp32 and the LSE in log2 units, rows in LSE order
// (b, h, i).  A row of D 16-bit values is D / 8 sixteen-byte chunks; each
// thread reads one chunk of O and dO for each of two rows (all four loads in
// flight together), and the D / 8 lanes of a row sum with shuffles.  A row
// without visible keys (LSE = -inf) gets +inf, so exp2(s - lse) = 0 for it.
constexpr int kRowsPerThread = 2;
template <int D, bool BF16>
__global__ void __launch_bounds__(256) fa_bwd_rows_kernel(const BwdParams p) {
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr int kLanes = D / 8;               // threads per row
  constexpr int kRowsPerBlock = 256 / kLanes;  // rows per pass of the block
  // block -> (batch * head, chunk of the head's rows): one 32-bit division
  const unsigned chunks = (unsigned)((p.Sq + kRowsPerThread * kRowsPerBlock - 1) /
                                     (kRowsPerThread * kRowsPerBlock));
  const unsigned bh = blockIdx.x / chunks, chunk = blockIdx.x - bh * chunks;
  const int b = (int)(bh / (unsigned)p.Hq), h = (int)(bh - (unsigned)b * p.Hq);
  const int sub = threadIdx.x % kLanes;
  float acc[kRowsPerThread];
  int64_t rid[kRowsPerThread];
  bool valid[kRowsPerThread];
  uint4 vo[kRowsPerThread], vg[kRowsPerThread];
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    const int i = (int)(chunk * kRowsPerThread + u) * kRowsPerBlock + threadIdx.x / kLanes;
    valid[u] = i < p.Sq;
    rid[u] = (int64_t)bh * p.Sq + i;
    vo[u] = vg[u] = make_uint4(0u, 0u, 0u, 0u);
    if (valid[u]) {
      const int64_t off = (((int64_t)b * p.Sq + i) * p.Hq + h) * D + sub * 8;
      vo[u] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const elem_t *>(p.o) + off);
      vg[u] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const elem_t *>(p.dout) + off);
    }
  }
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    const elem_t *eo = reinterpret_cast<const elem_t *>(&vo[u]);
    const elem_t *eg = reinterpret_cast<const elem_t *>(&vg[u]);
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) a += (float)eo[e] * (float)eg[e];
#pragma unroll
    for (int w = kLanes / 2; w > 0; w >>= 1) a += __shfl_xor_sync(0xffffffffu, a, w);
    acc[u] = a;
  }
#pragma unroll
  for (int u = 0; u < kRowsPerThread; ++u) {
    if (sub == 0 && valid[u]) {
      p.delta[rid[u]] = acc[u];
      const float l = p.lse[rid[u]];
      p.lse_l2[rid[u]] = (l == -INFINITY) ? INFINITY : l * 1.4426950408889634f;
    }
  }
}

// 32 fp32 values -> 16-bit, stored as four 16-byte chunks.
template <bool BF16>
__device__ __forceinline__ void store_row32(void *dst, const float *x, float mul) {
  uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
  for (int k = 0; k < 4; ++k)
    d[k] = make_uint4(pack_p<BF16>(x[8 * k] * mul, x[8 * k + 1] * mul),
                      pack_p<BF16>(x[8 * k + 2] * mul, x[8 * k + 3] * mul),
                      pack_p<BF16>(x[8 * k + 4] * mul, x[8 * k + 5] * mul),
                      pack_p<BF16>(x[8 * k + 6] * mul, x[8 * k + 7] * mul));
}

// SS MMA group: D[tmem] = A B^T over K = D, both operands K-major tiles.
template <int D>
__device__ __forceinline__ void issue_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  mma_ss(d, a, b, idesc, 0u);
#pragma unroll
  for (int kk = 1; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
    mma_ss_acc(d, a + off, b + off, idesc);
  }
}

// Half h of a TS MMA group: D[tmem] (+)= A[tmem] B over rows 64h .. 64h + 63
// of the B tile (four K = 16 steps); A is the half's 16-bit pairs in tensor-
// memory columns 64h .. 64h + 31 (the first half of the half's own 64 score
// columns, which only its own warpgroup reads), B an MN-major 128 x D tile.
// `accumulate` applies to the first step of half 0 (the group's first
// product).
__device__ __forceinline__ void issue_ts_half(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                              int h, bool accumulate) {
  const uint32_t ah = a + 64 * h;
  const uint64_t bh = b + ((h * 4 * 2048) >> 4);
  if (h == 0)
    mma_ts(d, ah, bh, idesc, accumulate ? 1u : 0u);
  else
    mma_ts_acc(d, ah, bh, idesc);
#pragma unroll
  for (int t = 1; t < 4; ++t) mma_ts_acc(d, ah + t * 8, bh + ((t * 2048) >> 4), idesc);
}

// Tensor-memory column (relative to a score tile) of the 16-bit pairs of
// score chunk c (32 columns): half c / 2 packs into the first 32 of its own
// 64 columns, so a warpgroup only overwrites columns it has read itself.
__device__ __forceinline__ uint32_t packed_col(int c) { return 64 * (c >> 1) + 16 * (c & 1); }

__device__ __forceinline__ void mul2(float &d0, float &d1, float a0, float a1, float b0,
                                     float b1) {
  const float2 d = __fmul2_rn(make_float2(a0, a1), make_float2(b0, b1));
  d0 = d.x;
  d1 = d.y;
}

// Key pass, 32 query columns 32c .. 32c + 31 of one key row: P^T = exp2(S^T
// scale log2e - lse) and dS^T = P^T (dP^T - Delta), written as 16-bit pairs
// over the columns already read.  MASKED: per-element visibility (a tile at
// a sequence end or crossing the causal diagonal); otherwise every element
// is visible.
template <bool BF16, bool MASKED, bool CAUSAL>
__device__ __forceinline__ void kv_chunk(uint32_t lane_base, int c, float sl2, const float *v_lse,
                                         const float *v_delta, int j, int q0, int Sq, int Sk,
                                         int off) {
  uint32_t sr[32], dr[32];
  tmem_ld32(lane_base + c * 32, sr);
  tmem_ld32(lane_base + 128 + c * 32, dr);
  tmem_wait_ld32(sr);
  tmem_wait_ld32(dr);
  const float2 *l2 = reinterpret_cast<const float2 *>(v_lse + c * 32);
  const float2 *dl = reinterpret_cast<const float2 *>(v_delta + c * 32);
  uint32_t pk[16], dk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float2 lv = l2[e], dv = dl[e];
    float x0, x1;
    fma_f32x2(x0, x1, __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), sl2, sl2,
              -lv.x, -lv.y);
    float p0 = ex2(x0), p1 = ex2(x1);
    float t0 = __uint_as_float(dr[2 * e]), t1 = __uint_as_float(dr[2 * e + 1]);
    add_f32x2(t0, t1, -dv.x, -dv.y);
    float d0, d1;
    mul2(d0, d1, p0, p1, t0, t1);
    if (MASKED) {  // selects, not products: a masked score may be inf or NaN
      const int qi = q0 + c * 32 + 2 * e;
      const bool ok_j = j < Sk;
      const bool v0 = ok_j && qi < Sq && (!CAUSAL || j <= qi + off);
      const bool v1 = ok_j && qi + 1 < Sq && (!CAUSAL || j <= qi + 1 + off);
      p0 = v0 ? p0 : 0.f;
      p1 = v1 ? p1 : 0.f;
      d0 = v0 ? d0 : 0.f;
      d1 = v1 ? d1 : 0.f;
    }
    pk[e] = pack_p<BF16>(p0, p1);
    dk[e] = pack_p<BF16>(d0, d1);
  }
  // P^T over S^T columns, dS^T over dP^T's, both in this chunk's half and
  // already read by this warp (chunk 2h + 1 packs over columns chunk 2h read)
  tmem_st16(lane_base + packed_col(c), pk);
  tmem_st16(lane_base + 128 + packed_col(c), dk);
}

// Query pass, 32 key columns 32c .. 32c + 31 of key tile kt for one query
// row: dS = exp2(S scale log2e - lse) (dP - Delta) as 16-bit pairs over S.
template <bool BF16, bool MASKED, bool CAUSAL>
__device__ __forceinline__ void q_chunk(uint32_t lane_base, uint32_t dp_off, int c, float sl2,
                                        float lse2, float dlt, int qi, int kt, int Sq, int Sk,
                                        int off) {
  uint32_t sr[32], dr[32];
  tmem_ld32(lane_base + c * 32, sr);
  tmem_ld32(lane_base + dp_off + c * 32, dr);
  tmem_wait_ld32(sr);
  tmem_wait_ld32(dr);
  uint32_t pk[16];
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    float x0, x1;
    fma_f32x2(x0, x1, __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]), sl2, sl2,
              -lse2, -lse2);
    float p0 = ex2(x0), p1 = ex2(x1);
    float t0 = __uint_as_float(dr[2 * e]), t1 = __uint_as_float(dr[2 * e + 1]);
    add_f32x2(t0, t1, -dlt, -dlt);
    float d0, d1;
    mul2(d0, d1, p0, p1, t0, t1);
    if (MASKED) {  // selects, not products: a masked score may be inf or NaN
      const int j = kt * kBlockN + c * 32 + 2 * e;
      const bool ok_q = qi < Sq;
      d0 = (ok_q && j < Sk && (!CAUSAL || j <= qi + off)) ? d0 : 0.f;
      d1 = (ok_q && j + 1 < Sk && (!CAUSAL || j + 1 <= qi + off)) ? d1 : 0.f;
    }
    pk[e] = pack_p<BF16>(d0, d1);
  }
  tmem_st16(lane_base + packed_col(c), pk);  // dS over S columns this warp read
}

// The sequence and 128-row tile of tile `idx` of a packed problem, counting
// every sequence's ceil(len / 128) tiles in order (lengths from the offsets
// cu[0 .. B]); {-1, 0} past the last tile.  Warp-collective: every lane of
// the calling warp gets the same result.
__device__ __forceinline__ int2 packed_tile(const int32_t *cu, int B, int idx, int lane) {
  int base = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int bb = b0 + lane;
    int cnt = 0;
    if (bb < B) {
      const int len = cu[bb + 1] - cu[bb];
      cnt = len > 0 ? (len + kBlockM - 1) / kBlockM : 0;
    }
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const int excl = incl - cnt;
    const unsigned m = __ballot_sync(0xffffffffu, bb < B && idx >= base + excl && idx < base + incl);
    if (m) {
      const int src = __ffs(m) - 1;
      return make_int2(b0 + src, idx - base - __shfl_sync(0xffffffffu, excl, src));
    }
    base += __shfl_sync(0xffffffffu, incl, 31);
  }
  return make_int2(-1, 0);
}

// Where a CTA's sequence lives: lengths, first token of its queries and keys
// in the tensors, and the batch coordinate of the tensor maps (dense: b;
// packed: 0, rows addressed by token).
struct SeqRef {
  int lq, lk, q_tok0, k_tok0, map_b;
};

__device__ __forceinline__ bool packed_seq(const BwdParams &p, int b, SeqRef *r) {
  const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
  if (q0 < 0 || q1 < q0 || q1 > p.Sq || k0 < 0 || k1 < k0 || k1 > p.Sk) return false;
  r->lq = q1 - q0;
  r->lk = k1 - k0;
  r->q_tok0 = q0;
  r->k_tok0 = k0;
  r->map_b = 0;
  return true;
}

// Zero rows [valid, 128) of a 128-row tile of D 16-bit columns in shared
// memory (whole 128-byte rows of each 64-column chunk, so the swizzle does
// not matter) and make the writes visible to the tensor core's proxy; the
// whole warp takes part.  A packed tile reaching past its sequence would
// otherwise feed the next sequence's rows (finite or not) into a product
// where 0 * inf = NaN.
template <int D>
__device__ __forceinline__ void zero_tail_rows(uint32_t tile, int valid, int lane) {
#pragma unroll 1
  for (int c = 0; c < D / 64; ++c)
#pragma unroll 1
    for (uint32_t o = (uint32_t)valid * 128u + lane * 16u; o < kChunkBytes; o += 512u)
      st_shared_v4(tile + c * kChunkBytes + o, 0u, 0u, 0u, 0u);
}

// ---------------------------------------------------------------- key pass
// Persistent: one CTA per SM walks a snake over the work items (key tile,
// batch, K/V head; heaviest key tiles first under causal masking; packed:
// every sequence's key tiles in order, K/V head fastest).  dV and dK of an
// item's 128 keys accumulate in tensor memory over every query tile that
// sees a key of the tile, for every query head of the group.  Across items
// the phases continue: the next item's K / V load starts once the previous
// item's last S^T / dP^T has read K / V, and its first dV / dK product waits
// until the previous item's accumulators are read out (acc_free), so the
// epilogue of one item overlaps the start of the next.
struct KvItem {
  int valid, b, g, k0, qt_begin, nq, n_it, off;
  SeqRef sq;
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ KvItem decode_kv_item(const BwdParams &p, int w, int lane) {
  KvItem t;
  t.valid = 0;
  t.sq = SeqRef{p.Sq, p.Sk, 0, 0, 0};
  int kt;
  if (VARLEN) {
    t.g = w % p.Hkv;
    const int2 bt = packed_tile(p.cu_k, p.B, w / p.Hkv, lane);
    if (bt.x < 0) return t;
    if (!packed_seq(p, bt.x, &t.sq)) {
      if (lane == 0) record_status(p.status, 5);
      return t;
    }
    t.b = bt.x;
    kt = bt.y;
  } else {
    const int bg = w % (p.B * p.Hkv);
    kt = w / (p.B * p.Hkv);
    t.b = bg / p.Hkv;
    t.g = bg % p.Hkv;
    t.sq.map_b = t.b;
  }
  t.k0 = kt * kBlockN;
  t.off = t.sq.lk - t.sq.lq;  // bottom-right aligned causal diagonal
  t.qt_begin = CAUSAL ? max(0, t.k0 - t.off) / kBlockM : 0;
  t.nq = max(0, (t.sq.lq + kBlockM - 1) / kBlockM - t.qt_begin);
  t.n_it = t.nq * p.group;
  t.valid = 1;
  return t;
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_kv_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = SmemBwd<D>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  const uint32_t kv_full = bar0, acc_ready = bar0 + 56, drain = bar0 + 64,
                 kv_empty = bar0 + 96, acc_free = bar0 + 104;
  // S^T / dP^T of queries 64h .. 64h + 63 computed (h = 0, 1)
  auto s_full = [&](int h) { return h ? bar0 + 112u : bar0 + 40u; };
  auto st_full = [&](int s) { return bar0 + 8u + 8u * s; };
  auto st_empty = [&](int s) { return bar0 + 24u + 8u * s; };
  // P^T / dS^T of queries 64h .. 64h + 63 written (h = 0, 1)
  auto p_half = [&](int h) { return h ? bar0 + 72u : bar0 + 48u; };
  // packed: stage s's query rows past the sequence zeroed
  auto st_fixed = [&](int s) { return bar0 + 80u + 8u * s; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);
  float *vec = reinterpret_cast<float *>(smem + L::kVecOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = VARLEN ? (p.k_tiles + p.B) * p.Hkv : p.k_tiles * p.B * p.Hkv;
  const int G = gridDim.x;
  auto item_of = [&](int i) {  // snake over the heavy-first item order
    return i * G + ((i & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(kv_full, 1);
    mbar_init(kv_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(st_full(s), 1);
      mbar_init(st_empty(s), 1);
      mbar_init(st_fixed(s), 1);
      mbar_init(p_half(s), 4);
    }
    mbar_init(s_full(0), 1);
    mbar_init(s_full(1), 1);
    mbar_init(acc_ready, 1);
    mbar_init(acc_free, 8);  // every elementwise warp, after reading dV / dK
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kBwdProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long limit = p.wait_limit;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return wait_bar(bar, par, abort_flag, limit, p.status);
  };
  // step s_ of item t: query head, first query row, tail past the sequence
  auto step_head = [&](const KvItem &t, int s_) { return t.g * p.group + s_ / t.nq; };
  auto step_q0 = [&](const KvItem &t, int s_) { return (t.qt_begin + s_ % t.nq) * kBlockM; };
  auto step_partial = [&](const KvItem &t, int s_) {
    return VARLEN && step_q0(t, s_) + kBlockM > t.sq.lq;
  };

  if (warp == kBwdProducer) {
    const uint64_t pol_res = policy_evict_first();
    const uint64_t pol_st = policy_evict_last();
    bool ok = true;
    int g_it = 0, n_acc = 0, issued = 0;
    for (int i = 0; ok; ++i) {
      const int w = item_of(i);
      if (w >= n_items) break;
      const KvItem t = decode_kv_item<CAUSAL, VARLEN>(p, w, lane);
      if (!t.valid || t.n_it == 0) continue;
      // the previous item's last S^T / dP^T has read K and V
      if (lane == 0 && n_acc > 0 && !wait(kv_empty, (n_acc - 1) & 1)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(kv_full, 2 * L::kTile);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sbase + L::kResOff + c * kChunkBytes, &tm_k, kv_full, c * 64, t.g,
                      t.sq.k_tok0 + t.k0, t.sq.map_b, pol_res);
          tma_load_4d(sbase + L::kResOff + L::kTile + c * kChunkBytes, &tm_v, kv_full, c * 64,
                      t.g, t.sq.k_tok0 + t.k0, t.sq.map_b, pol_res);
        }
      }
      ++n_acc;
      for (int s_ = 0; s_ < t.n_it && ok; ++s_, ++g_it) {
        const int s = g_it & 1;
        if (lane == 0 && g_it >= 2 && !wait(st_empty(s), ((g_it >> 1) - 1) & 1)) ok = false;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const int h = step_head(t, s_), q0 = step_q0(t, s_);
        const uint32_t dst = sbase + L::kStOff + s * 2 * L::kTile;
        if (lane == 0) {
          mbar_arrive_expect_tx(st_full(s), 2 * L::kTile);
          for (int c = 0; c < D / 64; ++c) {
            tma_load_4d(dst + c * kChunkBytes, &tm_q, st_full(s), c * 64, h, t.sq.q_tok0 + q0,
                        t.sq.map_b, pol_st);
            tma_load_4d(dst + L::kTile + c * kChunkBytes, &tm_do, st_full(s), c * 64, h,
                        t.sq.q_tok0 + q0, t.sq.map_b, pol_st);
          }
        }
        issued = g_it + 1;
        if (step_partial(t, s_)) {
          // rows past the sequence belong to the next one: zero them in Q and
          // dO (the B operands of dV += P^T dO and dK += dS^T Q) once landed
          ok = __all_sync(0xffffffffu, wait(st_full(s), (g_it >> 1) & 1));
          if (!ok) break;
          zero_tail_rows<D>(dst, t.sq.lq - q0, lane);
          zero_tail_rows<D>(dst + L::kTile, t.sq.lq - q0, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(st_fixed(s));
        }
      }
    }
    // drain the copies still in flight before the CTA exits (K / V loads are
    // serialised by kv_empty, so only the last can be outstanding)
    if (lane == 0 && n_acc > 0) {
      wait_bar(kv_full, (n_acc - 1) & 1, abort_flag, limit, p.status, false);
      for (int it = max(0, issued - 2); it < issued; ++it)
        wait_bar(st_full(it & 1), (it >> 1) & 1, abort_flag, limit, p.status, false);
    }
  } else if (warp == kBwdMma) {
    // the whole warp walks the items (the packed decode is warp-collective);
    // lane 0 issues every MMA and commit
    {
      constexpr uint32_t idesc_ss64 = make_idesc_f16(BF16, kBlockM, 64, false);
      constexpr uint32_t idesc_ts = make_idesc_f16(BF16, kBlockM, D, true);
      const uint64_t k_desc = make_sdesc_sw128(sbase + L::kResOff, 16, 1024);
      const uint64_t v_desc = make_sdesc_sw128(sbase + L::kResOff + L::kTile, 16, 1024);
      bool ok = true;
      int g_it = 0, n_acc = 0;
      uint32_t fixpar = 0;  // bit s: phase of st_fixed(s), as the producer counts it
      for (int i = 0; ok; ++i) {
        const int w = item_of(i);
        if (w >= n_items) break;
        const KvItem t = decode_kv_item<CAUSAL, VARLEN>(p, w, lane);
        if (!t.valid || t.n_it == 0) continue;
        if (lane == 0) {  // lanes 1-31 only follow the item sequence
          // Query halves are software-pipelined: per step it and half h the
          // issuer waits for P^T / dS^T of half h, issues dV += P^T dO and
          // dK += dS^T Q of that half, then the next step's S^T / dP^T of the
          // same half (N = 64), so one warpgroup's elementwise work overlaps
          // the products of the other half.  S^T / dP^T of a half overwrite
          // only that half's columns, whose packed P^T / dS^T the previous
          // products (earlier in issue order) have read.
          auto stage_ready = [&](int s_, int gs) {  // Q / dO of step s_ landed
            const int s = gs & 1;
            if (step_partial(t, s_)) {
              const bool r = wait(st_fixed(s), (fixpar >> s) & 1u);
              fixpar ^= 1u << s;
              return r;
            }
            return wait(st_full(s), (gs >> 1) & 1);
          };
          auto issue_scores = [&](int gs, int h) {  // S^T, dP^T of half h of step gs
            const uint32_t st = sbase + L::kStOff + (gs & 1) * 2 * L::kTile + h * 64 * 128;
            issue_ss<D>(tmem + 64 * h, k_desc, make_sdesc_sw128(st, 16, 1024), idesc_ss64);
            issue_ss<D>(tmem + 128 + 64 * h, v_desc,
                        make_sdesc_sw128(st + L::kTile, 16, 1024), idesc_ss64);
            tc_commit(s_full(h));
          };
          ok = wait(kv_full, n_acc & 1) && stage_ready(0, g_it);
          if (ok) {
            tc_fence_after();
            issue_scores(g_it, 0);
            issue_scores(g_it, 1);
            if (t.n_it == 1) tc_commit(kv_empty);  // K / V read for the last time
          }
          for (int s_ = 0; s_ < t.n_it && ok; ++s_, ++g_it) {
            const int s = g_it & 1;
            const uint32_t st = sbase + L::kStOff + s * 2 * L::kTile;
            const uint64_t do_mn = make_sdesc_sw128(st + L::kTile, kChunkBytes, 1024);
            const uint64_t q_mn = make_sdesc_sw128(st, kChunkBytes, 1024);
            const bool more = s_ + 1 < t.n_it;
            for (int hh = 0; hh < 2 && ok; ++hh) {
              ok = wait_bar_spin(p_half(hh), g_it & 1, abort_flag, limit, p.status);
              // the item's first product overwrites the accumulators: the
              // previous item's epilogue must have read them
              if (ok && s_ == 0 && hh == 0 && n_acc > 0) ok = wait(acc_free, (n_acc - 1) & 1);
              if (!ok) break;
              tc_fence_after();
              // dV += P^T dO, dK += dS^T Q (B tiles MN-major: rows = queries)
              issue_ts_half(tmem + 256, tmem, do_mn, idesc_ts, hh, s_ > 0);
              issue_ts_half(tmem + 256 + D, tmem + 128, q_mn, idesc_ts, hh, s_ > 0);
              if (hh == 1) tc_commit(st_empty(s));  // Q / dO of this step read
              if (more) {
                if (hh == 0) {
                  ok = stage_ready(s_ + 1, g_it + 1);
                  if (!ok) break;
                  tc_fence_after();
                }
                issue_scores(g_it + 1, hh);
                if (hh == 1 && s_ + 2 == t.n_it) tc_commit(kv_empty);
              }
            }
          }
          if (ok) {
            tc_commit(acc_ready);
            ++n_acc;
          }
        }  // lane 0
        ok = __shfl_sync(0xffffffffu, ok, 0);  // every lane, once per item
      }
      if (lane == 0) {
        // no MMA may still run when tensor memory is released
        tc_commit(drain);
        wait_bar(drain, 0, abort_flag, limit, p.status, false);
      }
    }
  } else {
    // -------------------------------------------- elementwise: one key per thread
    const int quarter = warp & 3, wg = warp >> 2;  // TMEM lane quarter, column half
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g_it = 0, n_acc = 0;
    for (int i = 0;; ++i) {
      const int w = item_of(i);
      if (w >= n_items) break;
      const KvItem t = decode_kv_item<CAUSAL, VARLEN>(p, w, lane);
      if (!t.valid) continue;
      const int lq = t.sq.lq, lk = t.sq.lk, k0 = t.k0, off = t.off;
      const int j = k0 + row;
      const int64_t lse_b = VARLEN ? 0 : (int64_t)t.b;
      const int64_t lse_row0 = VARLEN ? (int64_t)t.sq.q_tok0 : 0;
      // each warpgroup keeps lse / Delta of its own 64 queries (threads 0-63
      // of the warpgroup load them one step ahead, so the global-memory
      // latency overlaps the previous step's work); the warpgroups meet only
      // at their own named barrier, so their halves may run apart
      float n_lse = INFINITY, n_delta = 0.f;
      auto fetch = [&](int s_) {
        const int qi = step_q0(t, s_) + 64 * wg + row;
        const int64_t r = (lse_b * p.Hq + step_head(t, s_)) * p.Sq + lse_row0 + qi;
        n_lse = qi < lq ? p.lse_l2[r] : INFINITY;
        n_delta = qi < lq ? p.delta[r] : 0.f;
      };
      if (row < 64 && t.n_it > 0) fetch(0);
      for (int s_ = 0; s_ < t.n_it; ++s_, ++g_it) {
        const int s = g_it & 1;
        const int q0 = step_q0(t, s_);
        float *v_mine = vec + (2 * wg + s) * 128;  // [64 lse][64 Delta] of this half
        if (row < 64) {
          v_mine[row] = n_lse;
          v_mine[64 + row] = n_delta;
          if (s_ + 1 < t.n_it) fetch(s_ + 1);
        }
        named_barrier_sync(1 + wg, 128);
        // chunk c (32 queries) of this half reads entries (c - 2 wg) * 32 ..
        float *v_lse = v_mine - 64 * wg, *v_delta = v_mine + 64 - 64 * wg;
        if (ok) ok = __all_sync(0xffffffffu, wait(s_full(wg), g_it & 1));
        if (ok) {
          tc_fence_after();
          const bool interior = k0 + kBlockN <= lk && q0 + kBlockM <= lq &&
                                (!CAUSAL || k0 + kBlockN - 1 <= q0 + off);
#pragma unroll 1
          for (int c = 2 * wg; c < 2 * wg + 2; ++c) {
            if (interior)
              kv_chunk<BF16, false, CAUSAL>(lane_base, c, sl2, v_lse, v_delta, j, q0, lq, lk,
                                            off);
            else
              kv_chunk<BF16, true, CAUSAL>(lane_base, c, sl2, v_lse, v_delta, j, q0, lq, lk,
                                           off);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(p_half(wg));  // this half of the queries is written
        }
        __syncwarp();
      }
      // ----------------------------------------------------------- epilogue
      // Warpgroup wg owns columns wg D / 2 .. (wg + 1) D / 2 - 1 of dV and dK:
      // all of them are read out of tensor memory first and the accumulators
      // released (acc_free), then converted and stored through the warp's
      // staging buffer.  The loads are warp-wide (have, ok are warp-uniform);
      // only rows of keys inside the sequence are written.
      bool have = t.n_it > 0 && ok;
      if (have) have = __all_sync(0xffffffffu, wait(acc_ready, n_acc & 1));
      if (t.n_it > 0 && !have) ok = false;
      constexpr int kHalf = D / 2;
      uint32_t rv[kHalf], rk[kHalf];
      if (have) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c) {
          tmem_ld32(lane_base + 256 + wg * kHalf + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(rv + 32 * c));
          tmem_ld32(lane_base + 256 + D + wg * kHalf + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(rk + 32 * c));
        }
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c) {
          tmem_wait_ld32(*reinterpret_cast<uint32_t(*)[32]>(rv + 32 * c));
          tmem_wait_ld32(*reinterpret_cast<uint32_t(*)[32]>(rk + 32 * c));
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free);
      } else {
#pragma unroll
        for (int e = 0; e < kHalf; ++e) rv[e] = rk[e] = 0u;  // no query sees these keys
      }
      if (t.n_it > 0) ++n_acc;
      if (ok || t.n_it == 0) {  // warp-uniform
        // 32 columns of the warp's 32 key rows at a time: each lane packs its
        // row into the warp's staging buffer (16-byte pieces XOR-swizzled by
        // row, so neither side conflicts on banks), then the warp writes 8
        // whole 64-byte row pieces per store instead of 32 half sectors
        uint8_t *stg = smem + L::kEpiOff + warp * 2048;
        const int kr0 = k0 + quarter * 32;  // key of the warp's row 0
        const int64_t tok0 = lse_b * p.Sk + t.sq.k_tok0 + kr0;
#pragma unroll
        for (int which = 0; which < 2; ++which) {  // dV, then dK
          const uint32_t *src = which ? rk : rv;
          const float mul = which ? p.scale : 1.f;
          elem_t *out = reinterpret_cast<elem_t *>(which ? p.dk : p.dv);
#pragma unroll
          for (int c = 0; c < kHalf / 32; ++c) {
            const float *x = reinterpret_cast<const float *>(src + 32 * c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              *reinterpret_cast<uint4 *>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16)) =
                  make_uint4(pack_p<BF16>(x[8 * q] * mul, x[8 * q + 1] * mul),
                             pack_p<BF16>(x[8 * q + 2] * mul, x[8 * q + 3] * mul),
                             pack_p<BF16>(x[8 * q + 4] * mul, x[8 * q + 5] * mul),
                             pack_p<BF16>(x[8 * q + 6] * mul, x[8 * q + 7] * mul));
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int r = (lane >> 2) + 8 * k, pc = lane & 3;
              const uint4 v =
                  *reinterpret_cast<const uint4 *>(stg + r * 64 + ((pc ^ ((r >> 1) & 3)) * 16));
              if (kr0 + r < lk)
                *reinterpret_cast<uint4 *>(out + ((tok0 + r) * p.Hkv + t.g) * D + wg * kHalf +
                                           c * 32 + pc * 8) = v;
            }
            __syncwarp();
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// -------------------------------------------------------------- query pass
// Shared memory of the query pass: Q and dO resident, a three-slot K ring
// (S of key tile it + 2 is computed while dQ += dS K of tile it may still
// read K(it)) and a two-slot V ring.
template <int D>
struct SmemBwdQ {
  static constexpr uint32_t kTile = (D / 64) * kChunkBytes;
  static constexpr uint32_t kQOff = 0;
  static constexpr uint32_t kDoOff = kTile;
  static constexpr uint32_t kKOff = 2 * kTile;  // 3 slots
  static constexpr uint32_t kVOff = 5 * kTile;  // 2 slots
  static constexpr uint32_t kBarOff = 7 * kTile;
  // q_full, k_full[3], k_empty[3], v_full[2], v_empty[2], sdp_full,
  // ds_half[2], acc_ready, drain, k_fixed[3], q_empty, acc_free
  static constexpr int kNumBars = 21;
  static constexpr uint32_t kMiscOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kBytes = kMiscOff + 16;
  static constexpr uint32_t kAlloc = kBytes + 1024 > 120u * 1024 ? kBytes + 1024 : 120u * 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

// Persistent: one CTA per SM walks a snake over the work items (query tile,
// batch, query head; latest (heaviest) query tiles first under causal
// masking; packed: every sequence's query tiles in order, query head
// fastest).  dQ of an item's 128 rows accumulates in tensor memory over the
// key tiles the rows see.  The scores alternate between two tensor-memory
// buffers (columns 0-127 and 384-511; dP at 128-255, dQ at 256-383): per key
// tile the MMA issuer runs dP(it + 1), dQ += dS(it) K(it) and S(it + 2), so
// the elementwise work of tile it + 1 overlaps the last two.  Across items
// the key-tile counter and the K / V rings run on; the next item's Q / dO
// load starts once the item's last dP has read them, and its first dQ
// product waits until the previous dQ is read out (acc_free).
struct QItem {
  int valid, b, h, q0, n_kt, off, k_tiles;
  SeqRef sq;
};

template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ QItem decode_q_item(const BwdParams &p, int w, int lane) {
  QItem t;
  t.valid = 0;
  t.sq = SeqRef{p.Sq, p.Sk, 0, 0, 0};
  int qt;
  if (VARLEN) {
    t.h = w % p.Hq;
    const int2 bt = packed_tile(p.cu_q, p.B, w / p.Hq, lane);
    if (bt.x < 0) return t;
    if (!packed_seq(p, bt.x, &t.sq)) {
      if (lane == 0) record_status(p.status, 5);
      return t;
    }
    t.b = bt.x;
    qt = bt.y;
  } else {
    const int bh = w % (p.B * p.Hq);
    qt = p.q_tiles - 1 - w / (p.B * p.Hq);  // latest (heaviest) first
    t.b = bh / p.Hq;
    t.h = bh % p.Hq;
    t.sq.map_b = t.b;
  }
  t.q0 = qt * kBlockM;
  t.off = t.sq.lk - t.sq.lq;
  t.k_tiles = (t.sq.lk + kBlockN - 1) / kBlockN;
  t.n_kt = t.k_tiles;
  if (CAUSAL) {
    const int last = min(t.q0 + kBlockM, t.sq.lq) - 1 + t.off;  // last key any row sees
    t.n_kt = last < 0 ? 0 : min(t.k_tiles, last / kBlockN + 1);
  }
  t.valid = 1;
  return t;
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
__global__ void __launch_bounds__(kBwdThreads, 1)
    fa_bwd_q_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = SmemBwdQ<D>;
  using elem_t = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L::kBarOff;
  const uint32_t q_full = bar0, sdp_full = bar0 + 88, acc_ready = bar0 + 112,
                 drain = bar0 + 120, q_empty = bar0 + 152, acc_free = bar0 + 160;
  auto k_full = [&](int s) { return bar0 + 8u + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 32u + 8u * s; };
  auto v_full = [&](int s) { return bar0 + 56u + 8u * s; };
  auto v_empty = [&](int s) { return bar0 + 72u + 8u * s; };
  auto ds_half = [&](int hh) { return bar0 + 96u + 8u * hh; };
  // packed: K slot s's rows past the sequence's keys zeroed
  auto k_fixed = [&](int s) { return bar0 + 128u + 8u * s; };
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::kMiscOff);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::kMiscOff + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = VARLEN ? (p.q_tiles + p.B) * p.Hq : p.q_tiles * p.B * p.Hq;
  const int G = gridDim.x;
  auto item_of = [&](int i) {  // snake over the heavy-first item order
    return i * G + ((i & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < 3; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(k_fixed(s), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(ds_half(s), 4);
    }
    mbar_init(sdp_full, 1);
    mbar_init(acc_ready, 1);
    mbar_init(acc_free, 8);  // every elementwise warp, after reading dQ
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (warp == kBwdMma) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kBwdProducer && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const long long limit = p.wait_limit;
  auto wait = [&](uint32_t bar, uint32_t par) {
    return wait_bar(bar, par, abort_flag, limit, p.status);
  };
  // score buffer of global key-tile step gs
  auto s_buf = [&](int gs) { return (gs & 1) ? 384u : 0u; };

  if (warp == kBwdProducer) {
    const uint64_t pol_res = policy_evict_first();
    const uint64_t pol_st = policy_evict_last();
    bool ok = true;
    int gk = 0, n_acc = 0, k_issued = 0, v_issued = 0;
    for (int i = 0; ok; ++i) {
      const int w = item_of(i);
      if (w >= n_items) break;
      const QItem t = decode_q_item<CAUSAL, VARLEN>(p, w, lane);
      if (!t.valid || t.n_kt == 0) continue;
      // the previous item's last S and dP have read Q and dO
      if (lane == 0 && n_acc > 0 && !wait(q_empty, (n_acc - 1) & 1)) ok = false;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(q_full, 2 * L::kTile);
        for (int c = 0; c < D / 64; ++c) {
          tma_load_4d(sbase + L::kQOff + c * kChunkBytes, &tm_q, q_full, c * 64, t.h,
                      t.sq.q_tok0 + t.q0, t.sq.map_b, pol_res);
          tma_load_4d(sbase + L::kDoOff + c * kChunkBytes, &tm_do, q_full, c * 64, t.h,
                      t.sq.q_tok0 + t.q0, t.sq.map_b, pol_res);
        }
      }
      ++n_acc;
      const int g = t.h / p.group;
      for (int it = 0; it < t.n_kt && ok; ++it, ++gk) {
        const int ks = gk % 3, vs = gk & 1;
        if (lane == 0 && gk >= 3 && !wait(k_empty(ks), ((gk / 3) - 1) & 1)) ok = false;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        const uint32_t kdst = sbase + L::kKOff + ks * L::kTile;
        if (lane == 0) {
          mbar_arrive_expect_tx(k_full(ks), L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(kdst + c * kChunkBytes, &tm_k, k_full(ks), c * 64, g,
                        t.sq.k_tok0 + it * kBlockN, t.sq.map_b, pol_st);
        }
        k_issued = gk + 1;
        if (VARLEN && it * kBlockN + kBlockN > t.sq.lk) {
          // rows past the sequence's keys belong to the next one: zero them
          // in K (the B operand of dQ += dS K) once the tile has landed
          ok = __all_sync(0xffffffffu, wait(k_full(ks), (gk / 3) & 1));
          if (!ok) break;
          zero_tail_rows<D>(kdst, t.sq.lk - it * kBlockN, lane);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(k_fixed(ks));
        }
        if (lane == 0 && gk >= 2 && !wait(v_empty(vs), ((gk >> 1) - 1) & 1)) ok = false;
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(v_full(vs), L::kTile);
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sbase + L::kVOff + vs * L::kTile + c * kChunkBytes, &tm_v, v_full(vs),
                        c * 64, g, t.sq.k_tok0 + it * kBlockN, t.sq.map_b, pol_st);
        }
        v_issued = gk + 1;
      }
    }
    // drain the copies still in flight before the CTA exits (Q / dO loads
    // are serialised by q_empty, so only the last can be outstanding)
    if (lane == 0 && n_acc > 0) {
      wait_bar(q_full, (n_acc - 1) & 1, abort_flag, limit, p.status, false);
      for (int it = max(0, k_issued - 3); it < k_issued; ++it)
        wait_bar(k_full(it % 3), (it / 3) & 1, abort_flag, limit, p.status, false);
      for (int it = max(0, v_issued - 2); it < v_issued; ++it)
        wait_bar(v_full(it & 1), (it >> 1) & 1, abort_flag, limit, p.status, false);
    }
  } else if (warp == kBwdMma) {
    // the whole warp walks the items (the packed decode is warp-collective);
    // lane 0 issues every MMA and commit
    constexpr uint32_t idesc_ss = make_idesc_f16(BF16, kBlockM, kBlockN, false);
    constexpr uint32_t idesc_ts = make_idesc_f16(BF16, kBlockM, D, true);
    const uint64_t q_desc = make_sdesc_sw128(sbase + L::kQOff, 16, 1024);
    const uint64_t do_desc = make_sdesc_sw128(sbase + L::kDoOff, 16, 1024);
    auto k_addr = [&](int gs) { return sbase + L::kKOff + (gs % 3) * L::kTile; };
    auto v_addr = [&](int gs) { return sbase + L::kVOff + (gs & 1) * L::kTile; };
    bool ok = true;
    int gk = 0, n_acc = 0;
    uint32_t kfix = 0;  // bit s: phase of k_fixed(s), as the producer counts it
    for (int i = 0; ok; ++i) {
      const int w = item_of(i);
      if (w >= n_items) break;
      const QItem t = decode_q_item<CAUSAL, VARLEN>(p, w, lane);
      if (!t.valid || t.n_kt == 0) continue;
      if (lane == 0) {  // lanes 1-31 only follow the item sequence
        const int n = t.n_kt, g0 = gk;
        // S of item tile it (global step g0 + it) into its score buffer; a
        // partial packed tile is used once its tail rows are zeroed
        auto issue_s = [&](int it) {
          const int gs = g0 + it, ks = gs % 3;
          if (VARLEN && it * kBlockN + kBlockN > t.sq.lk) {
            if (!wait(k_fixed(ks), (kfix >> ks) & 1u)) return false;
            kfix ^= 1u << ks;
          } else if (!wait(k_full(ks), (gs / 3) & 1)) {
            return false;
          }
          tc_fence_after();
          issue_ss<D>(tmem + s_buf(gs), q_desc, make_sdesc_sw128(k_addr(gs), 16, 1024),
                      idesc_ss);
          return true;
        };
        // dP of item tile it = dO V^T; the V slot is released once it completes
        auto issue_dp = [&](int it) {
          const int gs = g0 + it;
          if (!wait(v_full(gs & 1), (gs >> 1) & 1)) return false;
          tc_fence_after();
          issue_ss<D>(tmem + 128, do_desc, make_sdesc_sw128(v_addr(gs), 16, 1024), idesc_ss);
          tc_commit(v_empty(gs & 1));
          return true;
        };
        ok = wait(q_full, n_acc & 1) && issue_s(0) && issue_dp(0);
        if (ok) {
          tc_commit(sdp_full);
          if (n == 1) tc_commit(q_empty);  // Q and dO read for the last time
          if (n > 1) ok = issue_s(1);
        }
        for (int it = 0; it < n && ok; ++it, ++gk) {
          // dS(it) written by both warpgroups (and S(it), dP(it) read)
          ok = wait_bar_spin(ds_half(0), gk & 1, abort_flag, limit, p.status) &&
               wait_bar_spin(ds_half(1), gk & 1, abort_flag, limit, p.status);
          if (!ok) break;
          tc_fence_after();
          if (it + 1 < n) {  // the next tile's dP first: its elementwise waits on it
            ok = issue_dp(it + 1);
            if (!ok) break;
            tc_commit(sdp_full);
            if (it + 2 == n) tc_commit(q_empty);  // the item's last dP (its last S is earlier)
          }
          // the item's first dQ product overwrites the accumulator: the
          // previous item's epilogue must have read it
          if (it == 0 && n_acc > 0) {
            ok = wait(acc_free, (n_acc - 1) & 1);
            if (!ok) break;
            tc_fence_after();
          }
          // dQ += dS(it) K(it) (K tile MN-major: rows = keys)
          const uint64_t k_mn = make_sdesc_sw128(k_addr(gk), kChunkBytes, 1024);
          issue_ts_half(tmem + 256, tmem + s_buf(gk), k_mn, idesc_ts, 0, it > 0);
          issue_ts_half(tmem + 256, tmem + s_buf(gk), k_mn, idesc_ts, 1, it > 0);
          tc_commit(k_empty(gk % 3));
          // S(it + 2) into the buffer dQ(it) reads (the pipe keeps issue order)
          if (it + 2 < n) ok = issue_s(it + 2);
        }
        if (ok) {
          tc_commit(acc_ready);
          ++n_acc;
        }
      }  // lane 0
      ok = __shfl_sync(0xffffffffu, ok, 0);  // every lane, once per item
    }
    if (lane == 0) {
      tc_commit(drain);
      wait_bar(drain, 0, abort_flag, limit, p.status, false);
    }
  } else {
    // ------------------------------------------ elementwise: one query row per thread
    const int quarter = warp & 3, wg = warp >> 2;  // TMEM lane quarter, column half
    const int row = quarter * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    int gk = 0, n_acc = 0;
    for (int i = 0;; ++i) {
      const int w = item_of(i);
      if (w >= n_items) break;
      const QItem t = decode_q_item<CAUSAL, VARLEN>(p, w, lane);
      if (!t.valid) continue;
      const int lq = t.sq.lq, lk = t.sq.lk, q0 = t.q0, off = t.off;
      const int qi = q0 + row;
      const int64_t lse_b = VARLEN ? 0 : (int64_t)t.b;
      const int64_t lse_row0 = VARLEN ? (int64_t)t.sq.q_tok0 : 0;
      const int64_t r = (lse_b * p.Hq + t.h) * p.Sq + lse_row0 + qi;
      const float lse2 = qi < lq ? p.lse_l2[r] : INFINITY;
      const float dlt = qi < lq ? p.delta[r] : 0.f;
      for (int it = 0; it < t.n_kt; ++it, ++gk) {
        if (ok) ok = __all_sync(0xffffffffu, wait(sdp_full, gk & 1));
        if (ok) {
          tc_fence_after();
          const bool interior = (it + 1) * kBlockN <= lk && q0 + kBlockM <= lq &&
                                (!CAUSAL || it * kBlockN + kBlockN - 1 <= q0 + off);
          const uint32_t base = lane_base + s_buf(gk);
          const uint32_t dp_minus_s = 128u - s_buf(gk);  // dP columns relative to base
#pragma unroll 1
          for (int c = 2 * wg; c < 2 * wg + 2; ++c) {
            if (interior)
              q_chunk<BF16, false, CAUSAL>(base, dp_minus_s, c, sl2, lse2, dlt, qi, it, lq, lk,
                                           off);
            else
              q_chunk<BF16, true, CAUSAL>(base, dp_minus_s, c, sl2, lse2, dlt, qi, it, lq, lk,
                                          off);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(ds_half(wg));  // this half of the keys is written
        }
        __syncwarp();
      }
      // ----------------------------------------------------------- epilogue
      // warpgroup wg reads columns wg D / 2 .. (wg + 1) D / 2 - 1 of dQ out of
      // tensor memory, releases the accumulator (acc_free), then stores
      bool have = t.n_kt > 0 && ok;
      if (have) have = __all_sync(0xffffffffu, wait(acc_ready, n_acc & 1));
      if (t.n_kt > 0 && !have) ok = false;
      constexpr int kHalf = D / 2;
      uint32_t rq[kHalf];
      if (have) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c)
          tmem_ld32(lane_base + 256 + wg * kHalf + c * 32,
                    *reinterpret_cast<uint32_t(*)[32]>(rq + 32 * c));
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c)
          tmem_wait_ld32(*reinterpret_cast<uint32_t(*)[32]>(rq + 32 * c));
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_free);
      } else {
#pragma unroll
        for (int e = 0; e < kHalf; ++e) rq[e] = 0u;  // the row sees no key
      }
      if (t.n_kt > 0) ++n_acc;
      if (qi < lq && (ok || t.n_kt == 0)) {
        elem_t *dq = reinterpret_cast<elem_t *>(p.dq) +
                     ((lse_b * p.Sq + t.sq.q_tok0 + qi) * p.Hq + t.h) * D + wg * kHalf;
#pragma unroll
        for (int c = 0; c < kHalf / 32; ++c)
          store_row32<BF16>(dq + c * 32, reinterpret_cast<const float *>(rq + 32 * c), p.scale);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kBwdMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool BF16, bool CAUSAL, bool VARLEN>
cudaError_t launch_bwd_t(const BwdLaunch &a) {
  const BwdParams &p = a.p;
  // the row pass sees a packed problem as one batch of Sq (= total) rows
  BwdParams pr = p;
  if (VARLEN) pr.B = 1;
  const int64_t rows = (int64_t)pr.B * pr.Hq * pr.Sq;
  if (rows > 0) {
    constexpr int64_t per_block = (int64_t)kRowsPerThread * 256 / (D / 8);
    const int64_t blocks = (int64_t)pr.B * pr.Hq * ((pr.Sq + per_block - 1) / per_block);
    if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
    fa_bwd_rows_kernel<D, BF16><<<(unsigned)blocks, 256, 0, a.stream>>>(pr);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  using L = SmemBwd<D>;
  using LQ = SmemBwdQ<D>;
  auto kv = fa_bwd_kv_kernel<D, BF16, CAUSAL, VARLEN>;
  auto qk = fa_bwd_q_kernel<D, BF16, CAUSAL, VARLEN>;
  static BwdOptIn opt_kv, opt_q;
  cudaError_t e = opt_kv.ensure(kv, (int)L::kAlloc, a.device);
  if (e != cudaSuccess) return e;
  e = opt_q.ensure(qk, (int)LQ::kAlloc, a.device);
  if (e != cudaSuccess) return e;
  // packed: every sequence rounds its tiles up once, so total / 128 + B
  // bounds the tiles; CTAs past the last one return at once
  const int64_t kv_ctas = VARLEN ? ((int64_t)p.k_tiles + p.B) * p.Hkv
                                 : (int64_t)p.k_tiles * p.B * p.Hkv;
  const int64_t q_ctas = VARLEN ? ((int64_t)p.q_tiles + p.B) * p.Hq
                                : (int64_t)p.q_tiles * p.B * p.Hq;
  if (kv_ctas > 0x7fffffffll || q_ctas > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  if (kv_ctas > 0) {
    // persistent: one CTA per SM walks the items
    const unsigned kv_grid = (unsigned)(kv_ctas < a.sms ? kv_ctas : a.sms);
    kv<<<kv_grid, kBwdThreads, L::kAlloc, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (q_ctas > 0) {
    const unsigned q_grid = (unsigned)(q_ctas < a.sms ? q_ctas : a.sms);
    qk<<<q_grid, kBwdThreads, LQ::kAlloc, a.stream>>>(a.tm_q, a.tm_k, a.tm_v, a.tm_do, p);
    e = cudaGetLastError();
  }
  return e;
}

template <int D, bool BF16>
cudaError_t launch_bwd_d(const BwdLaunch &a, bool causal, bool varlen) {
  if (causal)
    return varlen ? launch_bwd_t<D, BF16, true, true>(a) : launch_bwd_t<D, BF16, true, false>(a);
  return varlen ? launch_bwd_t<D, BF16, false, true>(a) : launch_bwd_t<D, BF16, false, false>(a);
}

}  // namespace

cudaError_t launch_bwd(const BwdLaunch &a, int D, bool bf16, bool causal, bool varlen) {
  if (D == 64)
    return bf16 ? launch_bwd_d<64, true>(a, causal, varlen)
                : launch_bwd_d<64, false>(a, causal, varlen);
  return bf16 ? launch_bwd_d<128, true>(a, causal, varlen)
              : launch_bwd_d<128, false>(a, causal, varlen);
}

}  // namespace fa
