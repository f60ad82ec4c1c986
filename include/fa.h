/*
 * fa.h — C ABI of the GB300 (sm_103a) exact attention forward library, libfa.so.
 *
 * The library computes, for every query row i of every (sequence b, query head
 * h), the exact softmax attention over the keys visible to that row:
 *
 *     s_ij  = scale * <q_i, k_j>
 *     O_i   = sum_j softmax(s_i)_j * v_j
 *     LSE_i = ln sum_j exp(s_ij)
 *
 * in one fused pass that streams K/V tiles through an online softmax with the
 * lazy rescale of the flash-attention fork's v1.7 release notes, section 1.2:
 * the running O and row_sum are rescaled only when the row max rises by more
 * than 8 log2 units, and on a skipped rescale the max stays at its previous
 * value ("max lagging"), so O, row_sum and P share one base and the result is
 * exact.  The upstream forward API it mirrors (flash_attn_func /
 * flash_attn_varlen_func with causal masking and grouped K/V heads) is listed
 * in the same notes, section 4.1; LSE is the [B, H, S] fp32 output of section
 * 4.6 (natural log).
 *
 * Every call is asynchronous on the given CUDA stream, allocates no device or
 * host memory, and is deterministic: two calls on the same inputs give
 * bit-identical O and LSE.
 *
 * All pointers are DEVICE pointers unless stated otherwise; the caller owns
 * every buffer.  A stream of NULL means the legacy default stream.
 */
#ifndef FA_H_
#define FA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t from cuda_runtime.h. */
typedef struct CUstream_st *fa_stream_t;

/* Status codes returned by the calls below. */
enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* a size, pointer, flag or alignment is invalid; nothing launched */
  FA_ERR_UNSUPPORTED = 2,  /* valid but not built (e.g. head dim other than 64, 128, 256)  */
  FA_ERR_CUDA = 3,         /* a CUDA runtime / driver call failed (no device, launch error) */
  FA_ERR_TIMEOUT = 4,      /* device: a pipeline wait exceeded its limit; outputs invalid    */
  FA_ERR_BAD_SEQLENS = 5,  /* device: cu_seqlens not monotone or beyond Sq / Sk; rows skipped */
  FA_ERR_SCRATCH_LIMIT = 6 /* fa_fwd_split_noalloc: the split scratch would exceed its fixed
                              buffer; nothing launched */
};

/* Element type of q, k, v and o. */
enum { FA_DTYPE_FP16 = 0, FA_DTYPE_BF16 = 1 };

/*
 * fa_fwd — exact attention forward (O and LSE).
 *
 * Layouts (row-major, contiguous, element type `dtype`):
 *   dense  (cu_seqlens_q == cu_seqlens_k == NULL):
 *     q, o  [B, Sq, Hq, D]     k, v  [B, Sk, Hkv, D]     lse [B, Hq, Sq] fp32
 *   packed variable-length (both cu_seqlens non-NULL):
 *     q, o  [Sq, Hq, D]        k, v  [Sk, Hkv, D]        lse [Hq, Sq]   fp32
 *     where Sq / Sk are the packed row counts (total query / key tokens) and
 *     cu_seqlens_q / cu_seqlens_k are int32 device arrays of B + 1 prefix
 *     offsets: sequence b owns q rows [cu_seqlens_q[b], cu_seqlens_q[b+1]) and
 *     k/v rows [cu_seqlens_k[b], cu_seqlens_k[b+1]).  Rows of q/o that belong
 *     to no sequence are neither read for any output nor written.  A
 *     sequence's output depends only on its own q/k/v rows: k/v rows of other
 *     sequences (or of none) may hold any values, Inf and NaN included (a
 *     tile reaching past a sequence's last key masks those keys and zeroes
 *     their v rows in shared memory before they are used).
 *
 * Arguments:
 *   q, k, v     inputs (16-byte aligned); k and v may be NULL when Sk == 0.
 *   o           output, same layout as q (16-byte aligned).
 *   lse         output log-sum-exp in natural-log units over the scaled scores,
 *               or NULL to skip it.  A row with no visible key gets O = 0 and
 *               LSE = -inf.
 *   B           batch size (dense) or number of sequences (packed); B = 0 is a
 *               no-op.
 *   Hq, Hkv     query / key-value heads; Hq % Hkv == 0 (grouped-query
 *               attention: query head h reads K/V head h / (Hq / Hkv)).
 *   Sq, Sk      sequence lengths (dense) or packed totals (packed), >= 0.
 *   D           head dimension: 64, 128 or 256.
 *   scale       score scale (commonly 1 / sqrt(D)); finite and > 0.
 *   causal      0 or 1.  With causal = 1 key j is visible to query i iff
 *               j <= i + (Lk - Lq) (diagonal aligned to the bottom-right; for
 *               Lq == Lk this is j <= i).
 *   stream      CUDA stream the work is queued on.
 *   dtype       FA_DTYPE_FP16 or FA_DTYPE_BF16.
 *
 * Returns FA_OK once the kernel is queued, or FA_ERR_INVALID_ARG /
 * FA_ERR_UNSUPPORTED (nothing queued) / FA_ERR_CUDA.  Errors found on the
 * device (FA_ERR_TIMEOUT, FA_ERR_BAD_SEQLENS) are recorded in a per-device
 * status word read by fa_get_device_error().
 */
int fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
           int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
           fa_stream_t stream, int dtype);

/*
 * fa_fwd_ex — fa_fwd with the score variants that the upstream forward API
 * offers next to plain causal masking (the fork's v1.7 release notes, section
 * 2 "Public APIs": local window, ALiBi, softcap; validated by tests 5-7 of
 * section 4.1 and the extra checks of section 4.6).  With window_left =
 * window_right = -1, softcap = 0 and alibi_slopes = NULL it is fa_fwd.
 *
 * All arguments of fa_fwd keep their meaning, layout and ownership.  Let
 * diag = i + (Lk - Lq) be the bottom-right aligned diagonal of query row i.
 *   window_left, window_right   local window: key j is visible to row i iff
 *               diag - window_left <= j <= diag + window_right; a negative
 *               bound is unbounded on that side.  causal = 1 additionally
 *               requires j <= diag.  Window (0, 0) with Lq == Lk leaves only
 *               key i, so O = V (section 4.6).
 *   softcap     0 (off) or a finite c > 0: each score becomes
 *               c * tanh(scale * <q_i, k_j> / c) before the softmax.
 *   alibi_slopes  NULL (off) or a DEVICE array of Hq fp32 slopes (4-byte
 *               aligned, read-only, finite): row i of query head h adds
 *               -alibi_slopes[h] * |diag - j| to each score (after the soft
 *               cap), natural-log units.
 * Every score is then combined in the same online softmax as fa_fwd (lazy
 * rescale, threshold 8 log2 units, max lagging); LSE is ln sum_j exp(score).
 * A row with no visible key gets O = 0 and LSE = -inf.
 *
 * Returns as fa_fwd; FA_ERR_INVALID_ARG also for a negative or non-finite
 * softcap (or one so small that scale / softcap overflows) and a misaligned
 * alibi_slopes.
 */
int fa_fwd_ex(const void *q, const void *k, const void *v, void *o, float *lse,
              int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
              const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
              fa_stream_t stream, int dtype,
              int window_left, int window_right, float softcap,
              const float *alibi_slopes);

/*
 * fa_fwd_split — fa_fwd_ex with the keys of every query tile split into
 * `num_splits` chunks processed by separate work units, each writing a
 * partial result (normalised O and LSE of its chunk), followed by an
 * LSE-weighted merge: M = max_s LSE_s, O = sum_s e^(LSE_s - M) O_s /
 * sum_s e^(LSE_s - M), LSE = M + ln sum_s e^(LSE_s - M).  This is the
 * split-KV forward of upstream FA2 (compute_attn_1rowblock_splitkv, one of
 * the dispatch sites in the fork's v1.2 notes, section 3); it fills the GPU
 * when a problem has fewer query tiles than streaming multiprocessors.  The
 * online softmax inside each chunk is the same as fa_fwd's (lazy rescale,
 * threshold 8 log2 units, max lagging; the chunk's first K/V tile sets its
 * max).  Each sequence's K/V tiles are cut into num_splits chunks of equal
 * tile count; a chunk a query row sees no key of contributes nothing.
 *
 * Arguments are those of fa_fwd_ex, plus:
 *   num_splits  1 = no split (same result as fa_fwd_ex); 2 .. 128 = that many
 *               chunks; 0 = chosen from the problem size and the number of
 *               multiprocessors (1 when the problem already fills the GPU).
 *
 * Scratch: with more than one split the call allocates
 * num_splits * rows * (D + 1) * 4 bytes of device memory (rows = number of
 * LSE entries) with cudaMallocAsync on `stream` and frees it with
 * cudaFreeAsync after the merge, both stream-ordered; the merge is a second
 * kernel on the same stream.  Returns as fa_fwd_ex; FA_ERR_INVALID_ARG also
 * for num_splits outside 0 .. 128, FA_ERR_CUDA if the scratch cannot be
 * allocated.
 */
int fa_fwd_split(const void *q, const void *k, const void *v, void *o, float *lse,
                 int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                 const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                 fa_stream_t stream, int dtype,
                 int window_left, int window_right, float softcap,
                 const float *alibi_slopes, int num_splits);

/*
 * fa_fwd_kvcache — attention of new query tokens over a KV cache, the
 * decoding path of the upstream API (flash_attn_with_kvcache, run as test 4
 * of the fork's v1.7 notes, section 4.1; paged KV caches per the upstream
 * survey and the FA4 changelog).  The cache is read as it is; this call does
 * not append to it.
 *
 * Layouts (element type `dtype`, row-major, contiguous):
 *   q, o      [B, Sq, Hq, D]   the Sq newest tokens of each sequence
 *   lse       [B, Hq, Sq] fp32 (natural log), or NULL
 *   contiguous cache (block_table == NULL):
 *     k_cache, v_cache  [B, page_rows, Hkv, D]: sequence b's keys are rows
 *     0 .. cache_seqlens[b]-1 of k_cache[b] (page_rows = cache capacity)
 *   paged cache (block_table != NULL):
 *     k_cache, v_cache  [num_pages, page_rows, Hkv, D]; block_table int32
 *     [B, max_blocks]: key j of sequence b is row j % page_rows of page
 *     block_table[b * max_blocks + j / page_rows]; page_rows must be a
 *     multiple of 128.
 *   cache_seqlens  int32 [B] (device): keys of each sequence, 0 ..
 *     capacity (page_rows without a table, max_blocks * page_rows with one).
 *     Cache rows past a sequence's length may hold any values, Inf and NaN
 *     included: they never reach the output.
 * Query token i of sequence b sits at position i + (cache_seqlens[b] - Sq)
 * of its sequence: causal = 1 makes key j visible iff j <= i +
 * cache_seqlens[b] - Sq (the bottom-right diagonal of fa_fwd).  window_left,
 * window_right, softcap and alibi_slopes are those of fa_fwd_ex; num_splits
 * those of fa_fwd_split (0 = chosen; scratch as documented there).
 *
 * Hq / Hkv must divide 128: the Hq / Hkv query heads of a K/V head are
 * processed together, so each K/V tile is read once for all of them.
 * Returns as fa_fwd; FA_ERR_INVALID_ARG also for page_rows <= 0, a paged
 * cache with max_blocks <= 0, num_pages <= 0 or page_rows not a multiple of
 * 128, or a NULL cache_seqlens; FA_ERR_UNSUPPORTED for Hq / Hkv not dividing
 * 128.  A cache_seqlens entry beyond the capacity, or a block_table entry
 * outside [0, num_pages), is reported as FA_ERR_BAD_SEQLENS by
 * fa_get_device_error (the affected outputs are not valid).
 */
int fa_fwd_kvcache(const void *q, const void *k_cache, const void *v_cache, void *o,
                   float *lse, int B, int Hq, int Hkv, int Sq, int D, float scale,
                   int causal, const int32_t *cache_seqlens, const int32_t *block_table,
                   int max_blocks, int page_rows, int num_pages, fa_stream_t stream,
                   int dtype, int window_left, int window_right, float softcap,
                   const float *alibi_slopes, int num_splits);

/*
 * fa_kvcache_plan — the split count fa_fwd_kvcache would use for these sizes
 * (capacity = cache keys a sequence can hold: page_rows without a block
 * table, max_blocks * page_rows with one) and its scratch bytes (written to
 * *scratch_bytes if non-NULL).  Returns the split count (>= 1) or minus a
 * status code.
 */
int fa_kvcache_plan(int B, int Hq, int Hkv, int Sq, int D, long long capacity,
                    int num_splits, long long *scratch_bytes);

/*
 * fa_fwd_split_noalloc — fa_fwd_split that allocates nothing.  It has no
 * counterpart in the pages: it exists for callers that must not allocate
 * device memory per call.  Arguments, results and status codes are those of
 * fa_fwd_split, computed by the same kernels.
 *
 * Scratch: instead of allocating, the split partials (num_splits * rows *
 * (D + 1) * 4 bytes, see fa_split_plan) live in one fixed device array of
 * fa_noalloc_scratch_bytes() bytes (32 MiB) inside the library, one per
 * device.  A call whose partials would not fit returns FA_ERR_SCRATCH_LIMIT
 * with nothing launched (pass a smaller num_splits, or use fa_fwd_split).
 * A call that needs no split (num_splits resolving to 1) does not touch the
 * array.  Nothing in the array has to start at zero: every partial slot the
 * merge reads is written by the same call first.
 *
 * The first call on a device that splits (after every argument check) looks
 * up the array's device address with cudaGetSymbolAddress (and fails with
 * FA_ERR_CUDA if that lookup fails); make that first call before any stream
 * capture.  Calls that may overlap in
 * time on one device (different streams, or different host threads) share
 * the array and race: their outputs are then undefined.  Serialise them on
 * one stream, or use fa_fwd_split.
 */
int fa_fwd_split_noalloc(const void *q, const void *k, const void *v, void *o, float *lse,
                         int B, int Hq, int Hkv, int Sq, int Sk, int D, float scale, int causal,
                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                         fa_stream_t stream, int dtype,
                         int window_left, int window_right, float softcap,
                         const float *alibi_slopes, int num_splits);

/* Size in bytes of the fixed scratch array of fa_fwd_split_noalloc. */
long long fa_noalloc_scratch_bytes(void);

/*
 * fa_split_plan — the split count fa_fwd_split would use for these sizes
 * (varlen: 1 for packed problems, where Sq / Sk are the packed totals) and
 * the device scratch it would allocate (bytes, written to *scratch_bytes if
 * non-NULL).  num_splits = 0 asks for the library's choice on the current
 * device.  Returns the split count (>= 1), or minus a status code.
 */
int fa_split_plan(int B, int Hq, int Hkv, int Sq, int Sk, int D, int varlen,
                  int num_splits, long long *scratch_bytes);

/*
 * fa_bwd — gradients of exact attention: the backward pass that the fork's
 * v1.7 release notes validate next to the forward (section 4.4), dense or
 * packed, head dim 64 or 128, fp16 or bf16.
 *
 * Inputs, all DEVICE memory in the layouts of fa_fwd:
 *   dense (cu_seqlens NULL):
 *     q [B, Sq, Hq, D], k / v [B, Sk, Hkv, D]  the forward's inputs
 *     o [B, Sq, Hq, D], lse [B, Hq, Sq] fp32    the forward's outputs (as
 *                                               fa_fwd with the same
 *                                               arguments wrote them)
 *     dout [B, Sq, Hq, D]                       dL/dO, the upstream gradient
 *   packed (cu_seqlens_q / cu_seqlens_k: B + 1 int32 offsets each, as in
 *   fa_fwd; Sq / Sk the token totals):
 *     q / o / dout [Sq, Hq, D], k / v [Sk, Hkv, D], lse [Hq, Sq]
 * Outputs (written in full, never accumulated into), the inputs' dtype:
 *   dq like q, dk / dv like k.
 * With P = softmax(scale q k^T) over each row's visible keys (causal masking
 * bottom-right aligned, as fa_fwd), dP = dout v^T and
 * dS = P * (dP - rowsum(dout * o)):
 *   dq = scale dS k,   dk = scale dS^T q,   dv = P^T dout,
 * dk and dv summed over the query heads of each K/V head's group.  Keys that
 * no query sees get zero gradients, rows without a visible key dq = 0.  The
 * result does not depend on scheduling (no atomics): repeated calls agree
 * bit for bit.
 *
 * Packed sequences may sit next to each other in any order of lengths; a
 * tile that reaches past its sequence reads the next one's rows, which may
 * hold any values (Inf and NaN included): they are masked and, where they
 * would feed a tensor-core product, zeroed in shared memory first.
 *
 * workspace: DEVICE memory owned by the caller, 16-byte aligned, at least
 * fa_bwd_workspace_bytes(B, Hq, Sq) bytes (packed: fa_bwd_workspace_bytes(1,
 * Hq, Sq) with Sq the total); used by this call's kernels on `stream` only
 * (two fp32 values per query row and head); contents on entry do not matter.
 *
 * Returns FA_OK once queued; FA_ERR_INVALID_ARG (nothing queued) for invalid
 * sizes, flags or scale, a NULL or misaligned pointer (16 bytes; lse and
 * cu_seqlens 4), only one cu_seqlens pointer, or a workspace smaller than
 * needed; FA_ERR_UNSUPPORTED for another head dim; FA_ERR_CUDA.  Recorded
 * on the device for fa_get_device_error: FA_ERR_TIMEOUT (a pipeline wait
 * timed out), FA_ERR_BAD_SEQLENS (offsets not monotone or past Sq / Sk).
 */
int fa_bwd(const void *q, const void *k, const void *v, const void *o, const float *lse,
           const void *dout, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int Sq,
           int Sk, int D, float scale, int causal, const int32_t *cu_seqlens_q,
           const int32_t *cu_seqlens_k, void *workspace, long long workspace_bytes,
           fa_stream_t stream, int dtype);

/* Device workspace fa_bwd needs for these sizes, in bytes (two fp32 values
 * per query row and head, 16-byte aligned halves), or minus a status code. */
long long fa_bwd_workspace_bytes(int B, int Hq, int Sq);

/*
 * fa_get_device_error — synchronize `stream`, then return and clear the status
 * word that kernels on the current device set on a device-side error
 * (FA_OK if none).  Returns FA_ERR_CUDA if the synchronization itself fails.
 */
int fa_get_device_error(fa_stream_t stream);

/*
 * fa_debug_wait_timeout — self-test of the bounded pipeline waits.  Launches
 * one block that waits on a shared-memory barrier nothing will ever arrive on,
 * once with the suspending wait and once with the polling wait of the MMA
 * issuers, each with a limit of `limit_cycles` SM clock cycles (1 .. 2^34).
 * When both give up as designed, FA_ERR_TIMEOUT is recorded in the device
 * status word (FA_ERR_INVALID_ARG if either wait misbehaved) and the kernel
 * returns normally; the context stays usable.  Returns the launch status.
 */
int fa_debug_wait_timeout(long long limit_cycles, fa_stream_t stream);

/*
 * fa_debug_trace_read — pipeline trace of a trace build (libfa_trace.so, built
 * with -DFA_TRACE).  The first CTA of every fa_fwd launch records SM clock64
 * stamps of its warp roles (softmax steps, MMA issue, TMA issue) into a
 * 2048-entry device buffer; this call synchronizes the device, copies the first
 * `n` entries (n <= 2048) to the HOST array `host_out` and clears the buffer.
 * Product builds return FA_ERR_UNSUPPORTED.
 */
int fa_debug_trace_read(unsigned long long *host_out, int n);

/*
 * fa_shutdown — forget the library's per-device state on every device.
 *
 * The library keeps, per device and created lazily by the first call there:
 * the device addresses of its status word and of the fixed scratch array of
 * fa_fwd_split_noalloc (both static device symbols of the library's module),
 * the multiprocessor count, and each kernel's opt-in to its large dynamic
 * shared memory.  It allocates no device or host memory, and tensor maps are
 * built per call, so there is nothing to free.  fa_shutdown() drops those
 * cached values; the next call on a device looks them up again.  Call it
 * after cudaDeviceReset() (which invalidates the cached addresses) or before
 * unloading the library.  It does not wait for queued work and must not run
 * while another host thread is inside a call of this library.  The pages
 * describe no such call: it belongs to this library's own lazily created
 * per-device state.  Returns FA_OK.
 */
int fa_shutdown(void);

/* Human-readable name of a status code (static string). */
const char *fa_status_string(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
