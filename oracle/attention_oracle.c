/*
 * CPU oracle for the exact attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline / reference leg may load or run this code.  It
 * shares nothing with the CUDA library: no headers, no helpers, no tables.
 *
 * Two functions, both in fp64, both over the same row addressing as the C ABI
 * (dense q/o [B, Sq, Hq, D], k/v [B, Sk, Hkv, D]; packed variable-length
 * q/o [total_q, Hq, D], k/v [total_k, Hkv, D] with cu_seqlens offsets):
 *
 *  oracle_attention()         the plain definition of attention: for one query
 *                             row, every visible score s_j = scale * <q, k_j>,
 *                             M = max s_j, l = sum exp(s_j - M),
 *                             O = sum exp(s_j - M) v_j / l, LSE = M + ln l.
 *                             Exact softmax attention as defined by the
 *                             FlashAttention papers and restated in the fork's
 *                             v1.7 release notes, section 1.2 ("output and LSE
 *                             stay exact").
 *
 *  oracle_attention_online()  the streaming (online-softmax) restatement of the
 *                             same result, walking 128-key blocks in ascending
 *                             order with the lazy-rescale rule of the v1.7
 *                             release notes, section 1.2 (skip the O / row_sum
 *                             rescale when scaled_diff >= -threshold, and on a
 *                             skip keep the previous row max: "max lagging"),
 *                             the Check_inf rule of the v1.2 release notes,
 *                             section 2 (a row max of -inf scales with 0), and
 *                             the exp2 formulation of scale_apply_exp2 (v1.2
 *                             release notes, section 2).  With lagging = 0 it
 *                             reproduces the superseded v1.2 behaviour (skip but
 *                             keep the new max), which is only used as a negative
 *                             control.  It counts skip / rescale events and the
 *                             largest P, which the v1.7 notes (section 1.2, "P
 *                             saturation") bound by exp2(8) = 256.
 *
 * Rows are addressed by their LSE index: dense rows by (b * Hq + h) * Sq + i,
 * packed rows by h * total_q + t (t = global token index).  Outputs are
 * written per requested row: o_rows[r * D + d], lse_rows[r].
 *
 *  oracle_attention_ex()      the same definition with the score variants the
 *                             fork's public API lists next to the plain forward
 *                             (v1.7 release notes, section 2 "Public APIs":
 *                             window, ALiBi, softcap; validated in section 4.1
 *                             tests 5-7 and section 4.6): a local window
 *                             (left, right), a tanh soft cap and ALiBi slopes.
 *                             oracle_attention() is this function with every
 *                             variant switched off.
 *
 *  oracle_attention_bwd()     the gradients of the plain definition (the
 *                             backward pass the fork's v1.7 release notes
 *                             validate in section 4.4): for a loss with
 *                             dL/dO = dO, per query row with its visible keys
 *                             P = softmax(S), S = scale * Q K^T,
 *                               dV_j += P_j dO,        dP_j = <dO, V_j>,
 *                               dS_j  = P_j (dP_j - sum_k P_k dP_k),
 *                               dQ    = scale * sum_j dS_j K_j,
 *                               dK_j += scale * dS_j Q,
 *                             the derivative of softmax written out (no
 *                             blocking, no recomputation tricks); K/V
 *                             gradients sum over the query heads of a group.
 *
 * Readings of points the pages leave open: LSE is the natural log over the
 * scaled scores; causal masking with Sq != Sk is aligned bottom-right (key j
 * visible iff j <= i + Lk - Lq); a row with no visible key gets O = 0 and
 * LSE = -inf.  For the variants, with
 * diag = i + Lk - Lq the bottom-right aligned diagonal of row i:
 *   window (left, right): key j visible iff diag - left <= j <= diag + right,
 *     a negative bound meaning unbounded on that side (so window (0, 0) with
 *     Sq = Sk leaves only key i and O = V[i], as section 4.6 reports); causal
 *     additionally requires j <= diag;
 *   softcap c > 0: s = c * tanh(scale * <q, k> / c);
 *   ALiBi: s gains -slope[h] * |diag - j| (natural-log units, after the soft
 *     cap), one slope per query head.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Locate the query row and its key range for one LSE index. */
typedef struct {
    int ok;
    int b, h, hkv;
    int64_t i;         /* row within its sequence                      */
    int64_t lq, lk;    /* query / key length of its sequence           */
    int64_t q_tok;     /* global token index of the query row          */
    int64_t k_tok0;    /* global token index of key 0 of the sequence  */
} row_ref;

static row_ref locate_row(int64_t id, int B, int Hq, int Hkv, int Sq, int Sk,
                          const int32_t *cu_q, const int32_t *cu_k) {
    row_ref r;
    memset(&r, 0, sizeof(r));
    const int group = Hq / Hkv;
    if (cu_q == NULL) {
        int64_t per_b = (int64_t)Hq * Sq;
        if (id < 0 || id >= (int64_t)B * per_b) return r;
        r.b = (int)(id / per_b);
        r.h = (int)((id / Sq) % Hq);
        r.i = id % Sq;
        r.lq = Sq;
        r.lk = Sk;
        r.q_tok = (int64_t)r.b * Sq + r.i;
        r.k_tok0 = (int64_t)r.b * Sk;
    } else {
        int64_t total_q = cu_q[B];
        if (id < 0 || id >= (int64_t)Hq * total_q) return r;
        r.h = (int)(id / total_q);
        int64_t t = id % total_q;
        int b = 0;
        while (b < B && !(cu_q[b] <= t && t < cu_q[b + 1])) b++;
        if (b == B) return r;
        r.b = b;
        r.i = t - cu_q[b];
        r.lq = cu_q[b + 1] - cu_q[b];
        r.lk = cu_k[b + 1] - cu_k[b];
        r.q_tok = t;
        r.k_tok0 = cu_k[b];
    }
    r.hkv = r.h / group;
    r.ok = 1;
    return r;
}

/* Number of visible keys of a row: keys 0 .. n-1 are visible. */
static int64_t visible_keys(const row_ref *r, int causal) {
    int64_t n = r->lk;
    if (causal) {
        int64_t last = r->i + r->lk - r->lq; /* bottom-right aligned diagonal */
        if (last + 1 < n) n = last + 1;
    }
    return n < 0 ? 0 : n;
}

/* Visible key range [*lo, *hi] of a row under causal masking and a local
 * window (negative bound = unbounded); returns the number of visible keys. */
static int64_t visible_range(const row_ref *r, int causal, int window_left,
                             int window_right, int64_t *lo, int64_t *hi) {
    const int64_t diag = r->i + r->lk - r->lq;
    int64_t a = 0, b = r->lk - 1;
    if (causal && diag < b) b = diag;
    if (window_right >= 0 && diag + window_right < b) b = diag + window_right;
    if (window_left >= 0 && diag - window_left > a) a = diag - window_left;
    *lo = a;
    *hi = b;
    return b >= a ? b - a + 1 : 0;
}

static int check_args(int B, int Hq, int Hkv, int Sq, int Sk, int D,
                      const int32_t *cu_q, const int32_t *cu_k) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if ((cu_q == NULL) != (cu_k == NULL)) return -1;
    return 0;
}

int oracle_attention_ex(const float *q, const float *k, const float *v,
                        double *o_rows, double *lse_rows,
                        int B, int Hq, int Hkv, int Sq, int Sk, int D,
                        double scale, int causal, int window_left, int window_right,
                        double softcap, const double *alibi_slopes,
                        const int32_t *cu_q, const int32_t *cu_k,
                        const int64_t *rows, int64_t nrows, int nthreads) {
    if (check_args(B, Hq, Hkv, Sq, Sk, D, cu_q, cu_k)) return -1;
    if (!(softcap >= 0.0)) return -1;
    int bad = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *s = NULL;
        int64_t s_cap = 0;
#pragma omp for schedule(dynamic, 8) reduction(| : bad)
        for (int64_t r = 0; r < nrows; r++) {
            row_ref ref = locate_row(rows[r], B, Hq, Hkv, Sq, Sk, cu_q, cu_k);
            double *out = o_rows + r * D;
            if (!ref.ok) { bad |= 1; continue; }
            int64_t j0, j1;
            int64_t n = visible_range(&ref, causal, window_left, window_right, &j0, &j1);
            if (n > s_cap) {
                free(s);
                s = (double *)malloc((size_t)n * sizeof(double));
                s_cap = n;
            }
            const float *qr = q + (ref.q_tok * Hq + ref.h) * (int64_t)D;
            const int64_t diag = ref.i + ref.lk - ref.lq;
            /* scores over the visible keys j0 .. j1: s = scale * <q, k_j>,
               then the soft cap, then the ALiBi distance penalty */
            double m = -INFINITY;
            for (int64_t c = 0; c < n; c++) {
                const int64_t j = j0 + c;
                const float *kr = k + ((ref.k_tok0 + j) * Hkv + ref.hkv) * (int64_t)D;
                double acc = 0.0;
                for (int d = 0; d < D; d++) acc += (double)qr[d] * (double)kr[d];
                double sc = scale * acc;
                if (softcap > 0.0) sc = softcap * tanh(sc / softcap);
                if (alibi_slopes) sc -= alibi_slopes[ref.h] * (double)llabs(diag - j);
                s[c] = sc;
                if (sc > m) m = sc;
            }
            for (int d = 0; d < D; d++) out[d] = 0.0;
            if (n == 0) { lse_rows[r] = -INFINITY; continue; }
            /* softmax weights relative to the row max, then O = P V / l */
            double l = 0.0;
            for (int64_t c = 0; c < n; c++) {
                double p = exp(s[c] - m);
                l += p;
                const float *vr = v + ((ref.k_tok0 + j0 + c) * Hkv + ref.hkv) * (int64_t)D;
                for (int d = 0; d < D; d++) out[d] += p * (double)vr[d];
            }
            for (int d = 0; d < D; d++) out[d] /= l;
            lse_rows[r] = m + log(l);
        }
        free(s);
    }
    return bad ? -2 : 0;
}

int oracle_attention(const float *q, const float *k, const float *v,
                     double *o_rows, double *lse_rows,
                     int B, int Hq, int Hkv, int Sq, int Sk, int D,
                     double scale, int causal,
                     const int32_t *cu_q, const int32_t *cu_k,
                     const int64_t *rows, int64_t nrows, int nthreads) {
    return oracle_attention_ex(q, k, v, o_rows, lse_rows, B, Hq, Hkv, Sq, Sk, D, scale,
                               causal, -1, -1, 0.0, NULL, cu_q, cu_k, rows, nrows,
                               nthreads);
}

int oracle_attention_online(const float *q, const float *k, const float *v,
                            double *o_rows, double *lse_rows,
                            int B, int Hq, int Hkv, int Sq, int Sk, int D,
                            double scale, int causal,
                            const int32_t *cu_q, const int32_t *cu_k,
                            const int64_t *rows, int64_t nrows,
                            int block_n, double threshold, int lagging,
                            int64_t *n_skip, int64_t *n_rescale, double *max_p,
                            int nthreads) {
    if (check_args(B, Hq, Hkv, Sq, Sk, D, cu_q, cu_k) || block_n <= 0) return -1;
    const double scale_log2 = scale * 1.4426950408889634074; /* scale * log2(e) */
    int bad = 0;
    int64_t skips = 0, rescales = 0;
    double pmax = 0.0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *t = (double *)malloc((size_t)block_n * sizeof(double));
#pragma omp for schedule(dynamic, 8) reduction(| : bad) reduction(+ : skips, rescales) reduction(max : pmax)
        for (int64_t r = 0; r < nrows; r++) {
            row_ref ref = locate_row(rows[r], B, Hq, Hkv, Sq, Sk, cu_q, cu_k);
            double *acc_o = o_rows + r * D;
            if (!ref.ok) { bad |= 1; continue; }
            int64_t n = visible_keys(&ref, causal);
            const float *qr = q + (ref.q_tok * Hq + ref.h) * (int64_t)D;
            for (int d = 0; d < D; d++) acc_o[d] = 0.0;
            double row_max = -INFINITY; /* raw (unscaled) score units */
            double row_sum = 0.0;
            int64_t nblocks = (n + block_n - 1) / block_n;
            for (int64_t blk = 0; blk < nblocks; blk++) {
                int64_t j0 = blk * block_n;
                int64_t cnt = n - j0 < block_n ? n - j0 : block_n;
                /* raw scores of this block and their max */
                double blk_max = -INFINITY;
                for (int64_t c = 0; c < cnt; c++) {
                    const float *kr = k + ((ref.k_tok0 + j0 + c) * Hkv + ref.hkv) * (int64_t)D;
                    double a = 0.0;
                    for (int d = 0; d < D; d++) a += (double)qr[d] * (double)kr[d];
                    t[c] = a;
                    if (a > blk_max) blk_max = a;
                }
                double cur_max = row_max > blk_max ? row_max : blk_max;
                if (blk == 0) {
                    row_max = cur_max; /* first block sets the max, no threshold */
                } else {
                    /* scaled_diff <= 0; -inf when the row was fully masked so far */
                    double scaled_diff = (cur_max == -INFINITY)
                                             ? 0.0
                                             : (row_max - cur_max) * scale_log2;
                    if (scaled_diff >= -threshold) {
                        skips++;
                        if (!lagging) row_max = cur_max; /* superseded behaviour */
                    } else {
                        double alpha = exp2(scaled_diff);
                        row_sum *= alpha;
                        for (int d = 0; d < D; d++) acc_o[d] *= alpha;
                        row_max = cur_max;
                        rescales++;
                    }
                }
                double max_scaled = (row_max == -INFINITY) ? 0.0 : row_max * scale_log2;
                for (int64_t c = 0; c < cnt; c++) {
                    double p = exp2(t[c] * scale_log2 - max_scaled);
                    if (p > pmax) pmax = p;
                    row_sum += p;
                    const float *vr = v + ((ref.k_tok0 + j0 + c) * Hkv + ref.hkv) * (int64_t)D;
                    for (int d = 0; d < D; d++) acc_o[d] += p * (double)vr[d];
                }
            }
            if (row_sum > 0.0) {
                for (int d = 0; d < D; d++) acc_o[d] /= row_sum;
                lse_rows[r] = (row_max * scale_log2 + log2(row_sum)) * 0.69314718055994530942;
            } else {
                for (int d = 0; d < D; d++) acc_o[d] = 0.0;
                lse_rows[r] = -INFINITY;
            }
        }
        free(t);
    }
    if (n_skip) *n_skip = skips;
    if (n_rescale) *n_rescale = rescales;
    if (max_p) *max_p = pmax;
    return bad ? -2 : 0;
}

/* Gradients of the plain definition (oracle_attention) with respect to q, k
 * and v for the upstream gradient dout (same layout as the output): dq has
 * q's layout, dk / dv have k's.  Parallel over (sequence, K/V head) groups,
 * each of which owns its dk / dv rows.  Rows without visible keys get dq = 0
 * and add nothing. */
int oracle_attention_bwd(const float *q, const float *k, const float *v, const float *dout,
                         double *dq, double *dk, double *dv,
                         int B, int Hq, int Hkv, int Sq, int Sk, int D,
                         double scale, int causal,
                         const int32_t *cu_q, const int32_t *cu_k, int nthreads) {
    if (check_args(B, Hq, Hkv, Sq, Sk, D, cu_q, cu_k)) return -1;
    const int group = Hq / Hkv;
    const int64_t total_q = cu_q ? (int64_t)cu_q[B] : (int64_t)B * Sq;
    const int64_t total_k = cu_k ? (int64_t)cu_k[B] : (int64_t)B * Sk;
    memset(dq, 0, (size_t)(total_q * Hq * D) * sizeof(double));
    memset(dk, 0, (size_t)(total_k * Hkv * D) * sizeof(double));
    memset(dv, 0, (size_t)(total_k * Hkv * D) * sizeof(double));
    int64_t max_lk = Sk;
    if (cu_k) {
        max_lk = 0;
        for (int b = 0; b < B; b++)
            if (cu_k[b + 1] - cu_k[b] > max_lk) max_lk = cu_k[b + 1] - cu_k[b];
    }
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
#pragma omp parallel
    {
        double *p = (double *)malloc((size_t)(max_lk > 0 ? max_lk : 1) * sizeof(double));
        double *dp = (double *)malloc((size_t)(max_lk > 0 ? max_lk : 1) * sizeof(double));
#pragma omp for schedule(dynamic, 1)
        for (int64_t gid = 0; gid < (int64_t)B * Hkv; gid++) {
            const int b = (int)(gid / Hkv), g = (int)(gid % Hkv);
            const int64_t lq = cu_q ? cu_q[b + 1] - cu_q[b] : Sq;
            const int64_t lk = cu_k ? cu_k[b + 1] - cu_k[b] : Sk;
            const int64_t q_tok0 = cu_q ? cu_q[b] : (int64_t)b * Sq;
            const int64_t k_tok0 = cu_k ? cu_k[b] : (int64_t)b * Sk;
            for (int h = g * group; h < (g + 1) * group; h++) {
                for (int64_t i = 0; i < lq; i++) {
                    int64_t n = lk;
                    if (causal && i + lk - lq + 1 < n) n = i + lk - lq + 1;
                    if (n <= 0) continue;
                    const float *qr = q + ((q_tok0 + i) * Hq + h) * (int64_t)D;
                    const float *dor = dout + ((q_tok0 + i) * Hq + h) * (int64_t)D;
                    double *dqr = dq + ((q_tok0 + i) * Hq + h) * (int64_t)D;
                    /* P = softmax of the scaled scores over the visible keys */
                    double m = -INFINITY;
                    for (int64_t j = 0; j < n; j++) {
                        const float *kr = k + ((k_tok0 + j) * Hkv + g) * (int64_t)D;
                        double acc = 0.0;
                        for (int d = 0; d < D; d++) acc += (double)qr[d] * (double)kr[d];
                        p[j] = scale * acc;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (int64_t j = 0; j < n; j++) {
                        p[j] = exp(p[j] - m);
                        l += p[j];
                    }
                    /* dP_j = <dO, V_j> and the row's sum_k P_k dP_k */
                    double delta = 0.0;
                    for (int64_t j = 0; j < n; j++) {
                        p[j] /= l;
                        const float *vr = v + ((k_tok0 + j) * Hkv + g) * (int64_t)D;
                        double acc = 0.0;
                        for (int d = 0; d < D; d++) acc += (double)dor[d] * (double)vr[d];
                        dp[j] = acc;
                        delta += p[j] * acc;
                    }
                    for (int64_t j = 0; j < n; j++) {
                        const double ds = p[j] * (dp[j] - delta);
                        const float *kr = k + ((k_tok0 + j) * Hkv + g) * (int64_t)D;
                        double *dkr = dk + ((k_tok0 + j) * Hkv + g) * (int64_t)D;
                        double *dvr = dv + ((k_tok0 + j) * Hkv + g) * (int64_t)D;
                        for (int d = 0; d < D; d++) {
                            dqr[d] += scale * ds * (double)kr[d];
                            dkr[d] += scale * ds * (double)qr[d];
                            dvr[d] += p[j] * (double)dor[d];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return 0;
}

/* Threads the oracle would use by default (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
