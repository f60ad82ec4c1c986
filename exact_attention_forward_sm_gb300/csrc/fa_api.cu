// C ABI of libfa.so: argument checks, TMA tensor maps, kernel dispatch and the
// per-device status word.  See include/fa.h for the contract of each call.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_bwd.cuh"
#include "fa_combine.cuh"
#include "fa_launch.cuh"

// Status word written by kernels on a device-side error (first error wins).
// Host code only ever uses its device address, fetched per device below.
__device__ int g_fa_status;

// Fixed split-KV scratch of fa_fwd_split_noalloc (that call allocates nothing;
// concurrent calls on one device share this array).
constexpr size_t kFixedScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_fa_fixed_scratch[kFixedScratchBytes];

#ifdef FA_TRACE
// Pipeline trace buffer of trace builds (see FA_TRACE_AT in the kernel).
__device__ unsigned long long g_fa_trace[fa::kTraceEntries];
#endif

namespace fa {

std::atomic<unsigned> &launch_epoch() {
  static std::atomic<unsigned> epoch{0};
  return epoch;
}

// Kernel used only to exercise the bounded waits: nothing arrives on the
// barrier.  The suspending wait (wait_bar) and the polling one of the MMA
// issuers (wait_bar_spin) each wait `limit` cycles; FA_ERR_TIMEOUT is recorded
// only if both gave up and recorded it themselves, anything else records
// FA_ERR_INVALID_ARG.
static __global__ void fa_wait_timeout_kernel(long long limit, int *status) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  __shared__ int local_status;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    local_status = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool got1 = wait_bar(smem_u32(&bar), 0, &abort_flag, limit, &local_status);
    const int st1 = local_status;
    abort_flag = 0;
    local_status = 0;
    const bool got2 = wait_bar_spin(smem_u32(&bar), 0, &abort_flag, limit, &local_status);
    const int st2 = local_status;
    record_status(status, (!got1 && !got2 && st1 == 4 && st2 == 4) ? 4 : 1);
  }
  __syncthreads();
}

}  // namespace fa

// Lazy-rescale threshold in log2 units (8 for 16-bit inputs); a build-time
// define so the threshold-0 ablation is a separate library.
#ifndef FA_RESCALE_THRESHOLD
#define FA_RESCALE_THRESHOLD 8.0f
#endif

namespace {

constexpr int kMaxDevices = 64;
constexpr long long kDefaultWaitLimit = 1ll << 33;  // ~4 s of SM clock

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

std::mutex g_status_mu;
int *g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

// Streaming multiprocessors of `device` (the persistent grid has one CTA each).
int sm_count(int device) {
  if (device < 0 || device >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_sm_count[device] &&
      cudaDeviceGetAttribute(&g_sm_count[device], cudaDevAttrMultiProcessorCount, device) !=
          cudaSuccess)
    g_sm_count[device] = 0;
  return g_sm_count[device];
}

// Device address of g_fa_status on the current device.
int *status_ptr(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[device]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa_status) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_status_ptr[device] = static_cast<int *>(ptr);
  }
  return g_status_ptr[device];
}

void *g_fixed_scratch[kMaxDevices] = {};

// Forget every cached per-device value (fa_shutdown).
void reset_device_caches() {
  std::lock_guard<std::mutex> lock(g_status_mu);
  for (int d = 0; d < kMaxDevices; ++d) {
    g_status_ptr[d] = nullptr;
    g_sm_count[d] = 0;
    g_fixed_scratch[d] = nullptr;
  }
  fa::launch_epoch().fetch_add(1, std::memory_order_acq_rel);
}

// Device address of g_fa_fixed_scratch on `device` (looked up once per device).
void *fixed_scratch_ptr(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_fixed_scratch[device]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_fa_fixed_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_fixed_scratch[device] = ptr;
  }
  return g_fixed_scratch[device];
}

// Trace builds: point the kernel at the trace buffer.
bool set_trace(fa::FwdParams &p) {
#ifdef FA_TRACE
  void *tr = nullptr;
  if (cudaGetSymbolAddress(&tr, g_fa_trace) != cudaSuccess) return false;
  p.trace = static_cast<unsigned long long *>(tr);
#else
  (void)p;
#endif
  return true;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Tensor map over a [batch, rows, heads, D] (or packed [rows, heads, D]) buffer,
// box = 128 rows x 64 elements of one head, 128-byte swizzle.  Out-of-range
// rows read as zero.
bool make_map(CUtensorMap *m, const void *base, bool bf16, int D, int heads, int64_t rows,
              int64_t batch, int box_heads = 1, int box_rows = 128, int box_cols = 64) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)heads, (cuuint64_t)rows,
                              (cuuint64_t)batch};
  const cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)heads * D * 2,
                                 (cuuint64_t)rows * heads * D * 2};
  // 64-column boxes (128-byte rows) take the 128-byte swizzle, 32-column
  // boxes (64-byte rows) the 64-byte one
  const cuuint32_t box[4] = {(cuuint32_t)box_cols, (cuuint32_t)box_heads, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
             const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

constexpr int kMaxSplits = 128;

// Split count for num_splits = 0: the smallest split count whose wave
// efficiency (units * s over whole waves of SMs) is within 85% of the best
// one, with at least one K/V tile per split.  Problems that already fill the
// GPU are not split.
int choose_splits(int64_t units, int64_t kv_tiles, int sms) {
  if (units <= 0 || sms <= 0 || units * 5 >= (int64_t)sms * 4) return 1;
  const int64_t max_s = std::min<int64_t>({(int64_t)kMaxSplits, kv_tiles, (int64_t)sms});
  if (max_s <= 1) return 1;
  auto eff = [&](int64_t s) {
    const int64_t work = units * s;
    const int64_t waves = (work + sms - 1) / sms;
    return (double)work / (double)(waves * sms);
  };
  double best = 0.0;
  for (int64_t s = 1; s <= max_s; ++s) best = std::max(best, eff(s));
  for (int64_t s = 1; s <= max_s; ++s)
    if (eff(s) >= 0.85 * best) return (int)s;
  return 1;
}

// Split count chosen for num_splits = 0 (sizes already validated).
int auto_splits(int B, int Hq, int Hkv, int Sq, int Sk, int D, bool varlen, int sms) {
  // head dim 256: one 128-row query tile per unit
  const bool pair_heads = D != 256 && ((Hq / Hkv) % 2) == 0;
  const int head_units = pair_heads ? Hq / 2 : Hq;
  const int rows_per_unit = (pair_heads || D == 256) ? fa::kBlockM : 2 * fa::kBlockM;
  const int64_t row_units = (Sq + rows_per_unit - 1) / rows_per_unit;
  // K/V tiles of a sequence: dense Sk, packed the mean length
  const int64_t per_seq = varlen ? (Sk + B - 1) / B : Sk;
  return choose_splits(row_units * head_units * (varlen ? 1 : B),
                       (per_seq + fa::kBlockN - 1) / fa::kBlockN, sms);
}

// The library's fixed split-KV scratch (fa_fwd_split_noalloc), used instead
// of a stream-ordered allocation.  Its device address is looked up only when
// a call really splits, after every argument has been checked.
struct FixedScratch {
  size_t bytes;
};

// Launch the attention kernel (`launch`) and, with more than one split, the
// combine that merges its partials; the split scratch is the caller's fixed
// buffer or a stream-ordered allocation freed after the combine.
template <class LaunchFn>
int run_split(fa::LaunchArgs &a, int splits, int64_t lse_rows, int D, bool bf16, void *o,
              float *lse, int B, int Hq, int Sq, const int32_t *cu_q, int sms,
              const FixedScratch *fixed, LaunchFn launch) {
  void *scratch = nullptr;
  if (splits > 1) {
    const size_t o_bytes = (size_t)splits * (size_t)lse_rows * (size_t)D * sizeof(float);
    const size_t l_bytes = (size_t)splits * (size_t)lse_rows * sizeof(float);
    char *base = nullptr;
    if (fixed) {
      if (o_bytes + l_bytes > fixed->bytes) return FA_ERR_SCRATCH_LIMIT;
      base = static_cast<char *>(fixed_scratch_ptr(a.device));
      if (!base) return FA_ERR_CUDA;
    } else {
      if (cudaMallocAsync(&scratch, o_bytes + l_bytes, a.stream) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
      }
      base = static_cast<char *>(scratch);
    }
    a.p.o_part = reinterpret_cast<float *>(base);
    a.p.lse_part = reinterpret_cast<float *>(base + o_bytes);
  }
  cudaError_t e = launch(a);
  if (e == cudaSuccess && splits > 1) {
    fa::CombineParams c;
    c.o_part = a.p.o_part;
    c.lse_part = a.p.lse_part;
    c.o = o;
    c.lse = lse;
    c.rows = lse_rows;
    c.num_splits = splits;
    c.B = B;
    c.Hq = Hq;
    c.Sq = Sq;
    c.cu_q = cu_q;
    e = fa::launch_combine(c, D, bf16, sms, a.stream);
  }
  if (scratch && cudaFreeAsync(scratch, a.stream) != cudaSuccess && e == cudaSuccess)
    e = cudaErrorUnknown;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// Shared body of fa_fwd, fa_fwd_ex, fa_fwd_split and fa_fwd_split_noalloc.
// Window bounds < 0 are unbounded; softcap 0 and alibi == nullptr switch those
// variants off; num_splits 1 = no split, 0 = choose; fixed != nullptr takes
// the split scratch from that buffer instead of allocating it.
int forward(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
            int Hkv, int Sq, int Sk, int D, float scale, int causal,
            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, fa_stream_t stream,
            int dtype, int window_left, int window_right, float softcap,
            const float *alibi_slopes, int num_splits, const FixedScratch *fixed = nullptr) {
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  // ---------------------------------------------------------- argument checks
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(softcap) || softcap < 0.f) return FA_ERR_INVALID_ARG;
  const float cap_k = softcap > 0.f ? scale / softcap : 0.f;
  if (!std::isfinite(cap_k)) return FA_ERR_INVALID_ARG;
  if (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)) return FA_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens_q != nullptr;
  if (varlen != (cu_seqlens_k != nullptr)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0) return FA_OK;  // no query rows
  if (!q || !o) return FA_ERR_INVALID_ARG;
  if (Sk > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;  // k / v unused when there are no keys
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o)) return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  if (varlen && ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
                 (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u)))
    return FA_ERR_INVALID_ARG;

  // Window bounds: negative = unbounded; a bound beyond Sq + Sk (no row is
  // that far from a key) is unbounded too.  Causal masking is the right bound
  // 0 intersected with any right bound >= 0.
  const int64_t span = (int64_t)Sq + Sk;
  int win_l = (window_left < 0 || window_left > span) ? -1 : window_left;
  int win_r = (window_right < 0 || window_right > span) ? -1 : window_right;
  if (causal) win_r = 0;

  const int group = Hq / Hkv;
  // head dim 256: one 128-row query tile per unit (tensor memory holds one
  // 256-column O accumulator next to its scores)
  const bool wide = D == 256;
  const bool pair_heads = !wide && (group % 2) == 0;
  const int head_units = pair_heads ? Hq / 2 : Hq;
  const int rows_per_unit = (pair_heads || wide) ? fa::kBlockM : 2 * fa::kBlockM;
  const int64_t row_units = (Sq + rows_per_unit - 1) / rows_per_unit;
  // packed problems: each sequence rounds its row count up once, so this
  // bounds the number of units; the kernel skips the ones past the last
  const int64_t base_units =
      varlen ? (row_units + B) * head_units : row_units * B * head_units;
  if (base_units <= 0 || base_units > 0x7fffffffll) return FA_ERR_UNSUPPORTED;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  int *status = status_ptr(device);
  const int sms = sm_count(device);
  if (!status || sms <= 0) return FA_ERR_CUDA;

  const int splits = num_splits ? num_splits : auto_splits(B, Hq, Hkv, Sq, Sk, D, varlen, sms);
  // the instances with score variants also carry the split-KV path
  const bool ext =
      win_l >= 0 || win_r > 0 || softcap > 0.f || alibi_slopes != nullptr || splits > 1;
  const bool plain_causal = !ext && win_r == 0;
  // the score variants that are on pick the instance (each carries only
  // their code)
  const int var = (softcap > 0.f ? fa::kVarCap : 0) | (alibi_slopes ? fa::kVarAlibi : 0);
  const int64_t units = base_units * splits;
  if (units > 0x7fffffffll) return FA_ERR_UNSUPPORTED;
  const int64_t lse_rows = (int64_t)Hq * Sq * (varlen ? 1 : B);
  // dense: persistent, one CTA per SM walking a snake over the heavy-first
  // unit order; packed: unit costs follow the sequence lengths, so one CTA per
  // unit and the hardware's in-order CTA dispatch balances them
  const int64_t grid = varlen ? units : (units < sms ? units : sms);

  fa::LaunchArgs a;
  const bool bf16 = dtype == FA_DTYPE_BF16;
  const int64_t q_rows = Sq, k_rows = Sk;
  const int64_t q_batch = varlen ? 1 : B, k_batch = varlen ? 1 : B;
  if (!make_map(&a.tm_q, q, bf16, D, Hq, q_rows, q_batch)) return FA_ERR_CUDA;
  // the prefill kernels store O in 32-column quarters, the head-dim-256
  // kernel in 64-column halves
  if (!make_map(&a.tm_o, o, bf16, D, Hq, q_rows, q_batch, 1, 128, wide ? 64 : 32))
    return FA_ERR_CUDA;
  if (Sk > 0) {
    if (!make_map(&a.tm_k, k, bf16, D, Hkv, k_rows, k_batch)) return FA_ERR_CUDA;
    if (!make_map(&a.tm_v, v, bf16, D, Hkv, k_rows, k_batch)) return FA_ERR_CUDA;
  } else {
    a.tm_k = a.tm_q;  // never read: no query tile visits a key tile
    a.tm_v = a.tm_q;
  }
  fa::FwdParams &p = a.p;
  p.o = o;
  p.lse = lse;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = group;
  p.pair_heads = pair_heads ? 1 : 0;
  p.head_units = head_units;
  p.rows_per_unit = rows_per_unit;
  p.dense_row_units = (int)row_units;
  p.rows_fastest = (!varlen && win_l < 0 && win_r < 0) ? 1 : 0;
  p.total_units = (int)units;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.threshold = FA_RESCALE_THRESHOLD;
  p.win_l = win_l;
  p.win_r = win_r;
  // with a right bound (causal included) a later row block sees at least as
  // many keys as an earlier one, up to the few rows whose right bound is cut
  // at the last key: schedule the later ones first
  p.reverse_rows = win_r >= 0 ? 1 : 0;
  p.cap_k = cap_k;
  p.cap_l2 = softcap * 1.4426950408889634f;
  p.alibi = alibi_slopes;
  p.num_splits = splits;
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.part_rows = lse_rows;
  p.cache_seqlens = nullptr;
  p.block_table = nullptr;
  p.max_blocks = p.page_rows = p.num_pages = 0;
  p.tok_per_tile = fa::kBlockM;
  p.tok_blocks = 0;
  p.wait_limit = kDefaultWaitLimit;
  p.status = status;
  p.trace = nullptr;
  fa::set_divisors(p);
  if (!set_trace(p)) return FA_ERR_CUDA;
  a.grid = (int)grid;
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.device = device;

  auto launch = [&](const fa::LaunchArgs &la) {
    if (wide) {
      if (ext)
        return bf16 ? fa::launch_ext_d256_bf16(la, varlen) : fa::launch_ext_d256_fp16(la, varlen);
      return bf16 ? fa::launch_d256_bf16(la, plain_causal, varlen)
                  : fa::launch_d256_fp16(la, plain_causal, varlen);
    }
    if (ext) {
      if (D == 64)
        return bf16 ? fa::launch_ext_d64_bf16(la, varlen, var) : fa::launch_ext_d64_fp16(la, varlen, var);
      return bf16 ? fa::launch_ext_d128_bf16(la, varlen, var) : fa::launch_ext_d128_fp16(la, varlen, var);
    }
    if (D == 64)
      return bf16 ? fa::launch_d64_bf16(la, plain_causal, varlen)
                  : fa::launch_d64_fp16(la, plain_causal, varlen);
    return bf16 ? fa::launch_d128_bf16(la, plain_causal, varlen)
                : fa::launch_d128_fp16(la, plain_causal, varlen);
  };
  return run_split(a, splits, lse_rows, D, bf16, o, lse, B, Hq, Sq, cu_seqlens_q, sms, fixed,
                   launch);
}

// Body of fa_fwd_kvcache (see include/fa.h).
int forward_kvcache(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                    int B, int Hq, int Hkv, int Sq, int D, float scale, int causal,
                    const int32_t *cache_seqlens, const int32_t *block_table, int max_blocks,
                    int page_rows, int num_pages, fa_stream_t stream, int dtype,
                    int window_left, int window_right, float softcap,
                    const float *alibi_slopes, int num_splits) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(softcap) || softcap < 0.f) return FA_ERR_INVALID_ARG;
  const float cap_k = softcap > 0.f ? scale / softcap : 0.f;
  if (!std::isfinite(cap_k)) return FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  if (page_rows <= 0) return FA_ERR_INVALID_ARG;
  const bool paged = block_table != nullptr;
  if (paged && (max_blocks <= 0 || num_pages <= 0 || page_rows % fa::kBlockN != 0))
    return FA_ERR_INVALID_ARG;
  if (paged && (reinterpret_cast<uintptr_t>(block_table) & 3u)) return FA_ERR_INVALID_ARG;
  if (alibi_slopes && (reinterpret_cast<uintptr_t>(alibi_slopes) & 3u)) return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  const int group = Hq / Hkv;
  if (group > fa::kBlockM || (fa::kBlockM % group) != 0) return FA_ERR_UNSUPPORTED;
  if (B == 0 || Sq == 0) return FA_OK;
  if (!q || !o || !k_cache || !v_cache || !cache_seqlens) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return FA_ERR_INVALID_ARG;
  if (lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cache_seqlens) & 3u) return FA_ERR_INVALID_ARG;

  const int64_t capacity = paged ? (int64_t)max_blocks * page_rows : page_rows;
  const int64_t span = (int64_t)Sq + capacity;
  int win_l = (window_left < 0 || window_left > span) ? -1 : window_left;
  int win_r = (window_right < 0 || window_right > span) ? -1 : window_right;
  if (causal) win_r = 0;

  const int tok_per_tile = fa::kBlockM / group;
  const int64_t tok_blocks = (Sq + tok_per_tile - 1) / tok_per_tile;
  const int64_t base_units = (int64_t)B * Hkv * tok_blocks;
  if (base_units > 0x7fffffffll) return FA_ERR_UNSUPPORTED;

  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  int *status = status_ptr(device);
  const int sms = sm_count(device);
  if (!status || sms <= 0) return FA_ERR_CUDA;
  // split rule of fa_kvcache_plan (capacity stands in for the device-side lengths)
  const int splits = num_splits ? num_splits
                                : choose_splits(base_units, (capacity + fa::kBlockN - 1) /
                                                                fa::kBlockN, sms);
  const int64_t units = base_units * splits;
  if (units > 0x7fffffffll) return FA_ERR_UNSUPPORTED;
  const int64_t lse_rows = (int64_t)B * Hq * Sq;

  fa::LaunchArgs a;
  const bool bf16 = dtype == FA_DTYPE_BF16;
  // q / o: tiles of (tok_per_tile tokens) x (group heads) starting at head hkv * group
  if (!make_map(&a.tm_q, q, bf16, D, Hq, Sq, B, group, tok_per_tile)) return FA_ERR_CUDA;
  if (!make_map(&a.tm_o, o, bf16, D, Hq, Sq, B, group, tok_per_tile)) return FA_ERR_CUDA;
  // cache: [pages, page_rows, Hkv, D] (contiguous cache: one page per sequence)
  const int64_t pages = paged ? num_pages : B;
  if (!make_map(&a.tm_k, k_cache, bf16, D, Hkv, page_rows, pages)) return FA_ERR_CUDA;
  if (!make_map(&a.tm_v, v_cache, bf16, D, Hkv, page_rows, pages)) return FA_ERR_CUDA;
  fa::FwdParams &p = a.p;
  p.o = o;
  p.lse = lse;
  p.cu_q = nullptr;
  p.cu_k = nullptr;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = (int)std::min<int64_t>(capacity, 0x7fffffff);
  p.group = group;
  p.pair_heads = 0;
  p.head_units = Hkv;
  p.rows_per_unit = tok_per_tile;
  p.dense_row_units = (int)tok_blocks;
  p.rows_fastest = 0;
  p.total_units = (int)units;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.threshold = FA_RESCALE_THRESHOLD;
  p.win_l = win_l;
  p.win_r = win_r;
  p.reverse_rows = 0;
  p.cap_k = cap_k;
  p.cap_l2 = softcap * 1.4426950408889634f;
  p.alibi = alibi_slopes;
  p.num_splits = splits;
  p.o_part = nullptr;
  p.lse_part = nullptr;
  p.part_rows = lse_rows;
  p.cache_seqlens = cache_seqlens;
  p.block_table = block_table;
  p.max_blocks = paged ? max_blocks : 1;
  p.page_rows = page_rows;
  p.num_pages = (int)pages;
  p.tok_per_tile = tok_per_tile;
  p.tok_blocks = (int)tok_blocks;
  p.wait_limit = kDefaultWaitLimit;
  p.status = status;
  p.trace = nullptr;
  fa::set_divisors(p);
  if (!set_trace(p)) return FA_ERR_CUDA;
  a.grid = (int)(units < sms ? units : sms);
  a.stream = reinterpret_cast<cudaStream_t>(stream);
  a.device = device;
  auto launch = [&](const fa::LaunchArgs &la) {
    if (D == 64) return bf16 ? fa::launch_kvc_d64_bf16(la) : fa::launch_kvc_d64_fp16(la);
    return bf16 ? fa::launch_kvc_d128_bf16(la) : fa::launch_kvc_d128_fp16(la);
  };
  return run_split(a, splits, lse_rows, D, bf16, o, lse, B, Hq, Sq, nullptr, sms, nullptr,
                   launch);
}

}  // namespace

extern "C" {

int fa_version(void) { return 100; }  // 0.1.0

const char *fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_TIMEOUT: return "device pipeline wait timed out";
    case FA_ERR_BAD_SEQLENS: return "cu_seqlens inconsistent with Sq / Sk";
    case FA_ERR_SCRATCH_LIMIT: return "split scratch larger than the fixed buffer";
    default: return "unknown status";
  }
}

int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
           int Hkv, int Sq, int Sk, int D, float scale, int causal,
           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, fa_stream_t stream,
           int dtype) {
  return forward(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, cu_seqlens_q,
                 cu_seqlens_k, stream, dtype, -1, -1, 0.f, nullptr, 1);
}

int fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
              int Hkv, int Sq, int Sk, int D, float scale, int causal,
              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, fa_stream_t stream,
              int dtype, int window_left, int window_right, float softcap,
              const float *alibi_slopes) {
  return forward(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, cu_seqlens_q,
                 cu_seqlens_k, stream, dtype, window_left, window_right, softcap, alibi_slopes,
                 1);
}

int fa_fwd_split(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                 int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, fa_stream_t stream,
                 int dtype, int window_left, int window_right, float softcap,
                 const float *alibi_slopes, int num_splits) {
  return forward(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, cu_seqlens_q,
                 cu_seqlens_k, stream, dtype, window_left, window_right, softcap, alibi_slopes,
                 num_splits);
}

int fa_fwd_split_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                         fa_stream_t stream, int dtype, int window_left, int window_right,
                         float softcap, const float *alibi_slopes, int num_splits) {
  FixedScratch fixed;
  fixed.bytes = kFixedScratchBytes;
  return forward(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, D, scale, causal, cu_seqlens_q,
                 cu_seqlens_k, stream, dtype, window_left, window_right, softcap, alibi_slopes,
                 num_splits, &fixed);
}

int fa_fwd_kvcache(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                   int B, int Hq, int Hkv, int Sq, int D, float scale, int causal,
                   const int32_t *cache_seqlens, const int32_t *block_table, int max_blocks,
                   int page_rows, int num_pages, fa_stream_t stream, int dtype,
                   int window_left, int window_right, float softcap,
                   const float *alibi_slopes, int num_splits) {
  return forward_kvcache(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Sq, D, scale, causal,
                         cache_seqlens, block_table, max_blocks, page_rows, num_pages, stream,
                         dtype, window_left, window_right, softcap, alibi_slopes, num_splits);
}

long long fa_noalloc_scratch_bytes(void) { return (long long)kFixedScratchBytes; }

long long fa_bwd_workspace_bytes(int B, int Hq, int Sq) {
  if (B < 0 || Hq <= 0 || Sq < 0) return -FA_ERR_INVALID_ARG;
  const long long rows = (long long)B * Hq * Sq;
  return 4 * ((rows + 3) / 4 * 4) + 4 * rows;  // lse in log2 units, then delta
}

int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Sq,
           int Sk, int D, float scale, int causal, const int32_t *cu_seqlens_q,
           const int32_t *cu_seqlens_k, void *workspace, long long workspace_bytes,
           fa_stream_t stream, int dtype) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return FA_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
  const bool varlen = cu_seqlens_q != nullptr;
  if (varlen != (cu_seqlens_k != nullptr)) return FA_ERR_INVALID_ARG;
  if (varlen && ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
                 (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u)))
    return FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
  if (B == 0) return FA_OK;
  const bool rows_q = Sq > 0, rows_k = Sk > 0;
  if (rows_q && (!q || !o || !dout || !dq || !lse || !workspace)) return FA_ERR_INVALID_ARG;
  if (rows_k && (!k || !v || !dk || !dv)) return FA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace))
    return FA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return FA_ERR_INVALID_ARG;
  // packed: Sq / Sk are the token totals and the workspace is sized as for
  // one batch of Sq rows
  const int rows_b = varlen ? 1 : B;
  const long long need = fa_bwd_workspace_bytes(rows_b, Hq, Sq);
  if (rows_q && workspace_bytes < need) return FA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t elem = 2;
  // no keys: dq = 0; no queries: dk = dv = 0
  if (!rows_k) {
    if (rows_q &&
        cudaMemsetAsync(dq, 0, (size_t)rows_b * Sq * Hq * D * elem, st) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  if (!rows_q) {
    if (cudaMemsetAsync(dk, 0, (size_t)rows_b * Sk * Hkv * D * elem, st) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, (size_t)rows_b * Sk * Hkv * D * elem, st) != cudaSuccess)
      return FA_ERR_CUDA;
    return FA_OK;
  }
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  int *status = status_ptr(device);
  if (!status) return FA_ERR_CUDA;
  const bool bf16 = dtype == FA_DTYPE_BF16;
  fa::BwdLaunch a;
  if (!make_map(&a.tm_q, q, bf16, D, Hq, Sq, rows_b) ||
      !make_map(&a.tm_do, dout, bf16, D, Hq, Sq, rows_b) ||
      !make_map(&a.tm_k, k, bf16, D, Hkv, Sk, rows_b) ||
      !make_map(&a.tm_v, v, bf16, D, Hkv, Sk, rows_b))
    return FA_ERR_CUDA;
  const long long rows = (long long)rows_b * Hq * Sq;
  fa::BwdParams &p = a.p;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.lse_l2 = static_cast<float *>(workspace);
  p.delta = static_cast<float *>(workspace) + (rows + 3) / 4 * 4;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.group = Hq / Hkv;
  p.scale = scale;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.q_tiles = (Sq + fa::kBlockM - 1) / fa::kBlockM;
  p.k_tiles = (Sk + fa::kBlockN - 1) / fa::kBlockN;
  p.wait_limit = kDefaultWaitLimit;
  p.status = status;
  a.stream = st;
  a.device = device;
  a.sms = sm_count(device);
  if (a.sms <= 0) return FA_ERR_CUDA;
  return fa::launch_bwd(a, D, bf16, causal != 0, varlen) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_shutdown(void) {
  reset_device_caches();
  return FA_OK;
}

int fa_split_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, int varlen, int num_splits,
                  long long *scratch_bytes) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || Hq % Hkv != 0) return -FA_ERR_INVALID_ARG;
  if (varlen != 0 && varlen != 1) return -FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return -FA_ERR_INVALID_ARG;
  if (D != 64 && D != 128 && D != 256) return -FA_ERR_UNSUPPORTED;
  int splits = num_splits;
  if (B == 0 || Sq == 0) {
    splits = 1;
  } else if (splits == 0) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return -FA_ERR_CUDA;
    const int sms = sm_count(device);
    if (sms <= 0) return -FA_ERR_CUDA;
    splits = auto_splits(B, Hq, Hkv, Sq, Sk, D, varlen != 0, sms);
  }
  if (scratch_bytes) {
    const long long rows = (long long)Hq * Sq * (varlen ? 1 : B);
    *scratch_bytes = splits > 1 ? (long long)splits * rows * (D + 1) * 4 : 0;
  }
  return splits;
}

int fa_kvcache_plan(int B, int Hq, int Hkv, int Sq, int D, long long capacity, int num_splits,
                    long long *scratch_bytes) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Hq % Hkv != 0 || capacity <= 0)
    return -FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > kMaxSplits) return -FA_ERR_INVALID_ARG;
  const int group = Hq / Hkv;
  if ((D != 64 && D != 128) || group > fa::kBlockM || fa::kBlockM % group != 0)
    return -FA_ERR_UNSUPPORTED;
  int splits = num_splits;
  if (B == 0 || Sq == 0) {
    splits = 1;
  } else if (splits == 0) {
    int device = 0;
    if (cudaGetDevice(&device) != cudaSuccess) return -FA_ERR_CUDA;
    const int sms = sm_count(device);
    if (sms <= 0) return -FA_ERR_CUDA;
    const int tok_per_tile = fa::kBlockM / group;
    const int64_t units = (int64_t)B * Hkv * ((Sq + tok_per_tile - 1) / tok_per_tile);
    splits = choose_splits(units, (capacity + fa::kBlockN - 1) / fa::kBlockN, sms);
  }
  if (scratch_bytes) {
    const long long rows = (long long)B * Hq * Sq;
    *scratch_bytes = splits > 1 ? (long long)splits * rows * (D + 1) * 4 : 0;
  }
  return splits;
}

int fa_get_device_error(fa_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  int *status = status_ptr(device);
  if (!status) return FA_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return FA_ERR_CUDA;
  if (value != 0 && cudaMemset(status, 0, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  return value;
}

int fa_debug_trace_read(unsigned long long *host_out, int n) {
#ifdef FA_TRACE
  if (!host_out || n < 0 || n > fa::kTraceEntries) return FA_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return FA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(host_out, g_fa_trace, n * sizeof(unsigned long long)) != cudaSuccess)
    return FA_ERR_CUDA;
  static const unsigned long long zeros[fa::kTraceEntries] = {};
  if (cudaMemcpyToSymbol(g_fa_trace, zeros, sizeof(zeros)) != cudaSuccess) return FA_ERR_CUDA;
  return FA_OK;
#else
  (void)host_out;
  (void)n;
  return FA_ERR_UNSUPPORTED;
#endif
}

int fa_debug_wait_timeout(long long limit_cycles, fa_stream_t stream) {
  if (limit_cycles < 1 || limit_cycles > (1ll << 34)) return FA_ERR_INVALID_ARG;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess) return FA_ERR_CUDA;
  int *status = status_ptr(device);
  if (!status) return FA_ERR_CUDA;
  fa::fa_wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_cycles,
                                                                                   status);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
