/*
 * Causal grouped-query attention, plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. This is the slow, obviously correct definition
 * that the GPU library is checked against. Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference leg load it. The
 * product path never calls it, and it shares no code, header, table or
 * constant with the CUDA sources (neither side includes the other).
 *
 * What it computes. The step is the causal grouped-query attention of the
 * Qwen text encoder's prefill, layer 0, named in antirez/h3.c issue #47
 * ("Qwen layer 0 causal GQA failed: causal attention sequence 10231 exceeds
 * threadgroup memory", sections "Error" and "Suggested fix directions"):
 * every query row builds its causal attention score row over the keys at or
 * before its own position, normalises it with a softmax, and takes the
 * weighted sum of the value rows. Written out in fp64:
 *
 *   for each sequence b with token rows [s_b, e_b) (from cu_seqlens),
 *   for each query head h, its key/value head g = floor(h * Hkv / Hq),
 *   for each query row i in [s_b, e_b):
 *     z_j   = scale * sum_d q[h,i,d] * k[g,j,d]      for j in [s_b, i]
 *     m     = max_j z_j
 *     L     = m + ln( sum_j exp(z_j - m) )            (natural-log LSE)
 *     o[h,i,:] = sum_j exp(z_j - L) * v[g,j,:]
 *     lse[h,i] = L
 *
 * The bidirectional form (causal = 0) is the same sum over every key of the
 * sequence, j in [s_b, e_b): the long DiT attention that the h3.c README
 * ("Metal 4 and TensorOps paths") keeps on MPSGraph and whose 19316- and
 * 34121-row forwards tgo-app-dev/vpipe issue #10 reports.
 *
 * Readings where the pages are silent (they give no head mapping, scale,
 * layout or LSE convention):
 *   - contiguous head groups, g = h / (Hq/Hkv) (same as repeating each KV
 *     head Hq/Hkv times in place);
 *   - key j is visible to query i iff j <= i, positions counted from the
 *     start of each packed sequence; sequences never see each other;
 *   - the scale multiplies the logits (it is not folded into q);
 *   - LSE is the natural log of the sum of exp of the scaled logits;
 *   - layouts are head-major: q,o [Hq][T][D]; k,v [Hkv][T][D]; lse [Hq][T].
 *
 * Inputs arrive as raw bf16 bit patterns (uint16) and are widened exactly
 * to double. Everything after that is fp64. m is subtracted only to keep
 * exp() in range; the result is the plain definition above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact widening of one bf16 bit pattern: bf16 is the top half of an
 * IEEE-754 binary32, so shifting it into the high 16 bits gives the same
 * number as a float, and float -> double is exact. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Index of the packed sequence that holds token row t: the b with
 * cu[b] <= t < cu[b+1]. Zero-length sequences never hold a row. */
static int sequence_of(const int32_t *cu, int n_seqs, int64_t t)
{
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

static int check_args(const int32_t *cu, int n_seqs, int hq, int hkv, int d)
{
    if (!cu || n_seqs < 1 || hq < 1 || hkv < 1 || d < 1) return 1;
    if (hq % hkv != 0) return 2;
    if (cu[0] != 0) return 3;
    for (int b = 0; b < n_seqs; ++b)
        if (cu[b + 1] < cu[b]) return 4;
    return 0;
}

/* One query row (h, i): fills o_row[0..D) and *lse, and optionally the
 * probability row p_row[0..i-s_b] = exp(z_j - L). z is caller scratch of at
 * least (i - s_b + 1) doubles; qrow of D doubles. */
static void one_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const int32_t *cu, int n_seqs, int hq, int hkv, int d,
                    double scale, int causal, int64_t T, int h, int64_t i,
                    double *z, double *qrow, double *o_row, double *lse,
                    double *p_row)
{
    const int b = sequence_of(cu, n_seqs, i);
    const int64_t s_b = cu[b];
    const int64_t e_b = cu[b + 1];
    const int g = (int)(((int64_t)h * hkv) / hq);
    const int64_t n_causal = i - s_b + 1;          /* keys s_b .. i */
    const int64_t n = causal ? n_causal : e_b - s_b;

    for (int c = 0; c < d; ++c)
        qrow[c] = bf16_bits_to_double(q[((int64_t)h * T + i) * d + c]);

    /* logits of the causal score row */
    double m = -INFINITY;
    for (int64_t jj = 0; jj < n; ++jj) {
        const uint16_t *krow = k + ((int64_t)g * T + s_b + jj) * d;
        double dot = 0.0;
        for (int c = 0; c < d; ++c)
            dot += qrow[c] * bf16_bits_to_double(krow[c]);
        z[jj] = scale * dot;
        if (z[jj] > m) m = z[jj];
    }

    /* log-sum-exp of the row */
    double sum = 0.0;
    for (int64_t jj = 0; jj < n; ++jj)
        sum += exp(z[jj] - m);
    const double L = m + log(sum);

    /* softmax-weighted sum of the value rows */
    for (int c = 0; c < d; ++c) o_row[c] = 0.0;
    for (int64_t jj = 0; jj < n; ++jj) {
        const double p = exp(z[jj] - L);
        if (p_row) p_row[jj] = p;
        const uint16_t *vrow = v + ((int64_t)g * T + s_b + jj) * d;
        for (int c = 0; c < d; ++c)
            o_row[c] += p * bf16_bits_to_double(vrow[c]);
    }
    *lse = L;
}

static int64_t longest_sequence(const int32_t *cu, int n_seqs)
{
    int64_t best = 0;
    for (int b = 0; b < n_seqs; ++b)
        if (cu[b + 1] - cu[b] > best) best = cu[b + 1] - cu[b];
    return best;
}

/* Every row of every head: o [Hq][T][D], lse [Hq][T], both fp64; causal
 * selects the causal (1) or bidirectional (0) key range.
 * n_threads <= 0 keeps the OpenMP default. Returns 0 on success. */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const int32_t *cu_seqlens, int n_seqs,
                     int n_q_heads, int n_kv_heads, int head_dim, double scale,
                     int causal, double *o, double *lse, int n_threads)
{
    int rc = check_args(cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim);
    if (rc) return rc;
    const int64_t T = cu_seqlens[n_seqs];
    const int64_t smax = longest_sequence(cu_seqlens, n_seqs);
    const int64_t total = (int64_t)n_q_heads * T;
    if (total == 0) return 0;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(smax > 0 ? smax : 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!z || !qrow) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 8)
            for (int64_t r = 0; r < total; ++r) {
                const int h = (int)(r / T);
                const int64_t i = r % T;
                one_row(q, k, v, cu_seqlens, n_seqs, n_q_heads, n_kv_heads,
                        head_dim, scale, causal, T, h, i, z, qrow,
                        o + r * head_dim, lse + r, NULL);
            }
        }
        free(z);
        free(qrow);
    }
    return failed ? 5 : 0;
}

/* A chosen set of rows: rows[2*r] = query head h, rows[2*r+1] = token row t.
 * o_rows [n_rows][D], lse_rows [n_rows], fp64. Returns 0 on success. */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          const int32_t *cu_seqlens, int n_seqs,
                          int n_q_heads, int n_kv_heads, int head_dim, double scale,
                          int causal, const int64_t *rows, int64_t n_rows,
                          double *o_rows, double *lse_rows, int n_threads)
{
    int rc = check_args(cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim);
    if (rc) return rc;
    const int64_t T = cu_seqlens[n_seqs];
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= n_q_heads || rows[2 * r + 1] < 0 ||
            rows[2 * r + 1] >= T)
            return 6;
    const int64_t smax = longest_sequence(cu_seqlens, n_seqs);
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int failed = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(smax > 0 ? smax : 1));
        double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!z || !qrow) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t r = 0; r < n_rows; ++r)
                one_row(q, k, v, cu_seqlens, n_seqs, n_q_heads, n_kv_heads,
                        head_dim, scale, causal, T, (int)rows[2 * r], rows[2 * r + 1],
                        z, qrow, o_rows + r * head_dim, lse_rows + r, NULL);
        }
        free(z);
        free(qrow);
    }
    return failed ? 5 : 0;
}

/* The causal entry points: the definition above with causal = 1. */
int oracle_causal_gqa(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      const int32_t *cu_seqlens, int n_seqs,
                      int n_q_heads, int n_kv_heads, int head_dim, double scale,
                      double *o, double *lse, int n_threads)
{
    return oracle_attention(q, k, v, cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim,
                            scale, 1, o, lse, n_threads);
}

int oracle_causal_gqa_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                           const int32_t *cu_seqlens, int n_seqs,
                           int n_q_heads, int n_kv_heads, int head_dim, double scale,
                           const int64_t *rows, int64_t n_rows,
                           double *o_rows, double *lse_rows, int n_threads)
{
    return oracle_attention_rows(q, k, v, cu_seqlens, n_seqs, n_q_heads, n_kv_heads,
                                 head_dim, scale, 1, rows, n_rows, o_rows, lse_rows, n_threads);
}

/* The probability row of one query (h, t): p_out[j - s_b] = exp(z_j - L) for
 * j in [s_b, t]. Returns the row length (t - s_b + 1), or -1 on bad input. */
int64_t oracle_attention_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                               const int32_t *cu_seqlens, int n_seqs,
                               int n_q_heads, int n_kv_heads, int head_dim, double scale,
                               int h, int64_t t, double *p_out)
{
    if (check_args(cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim)) return -1;
    const int64_t T = cu_seqlens[n_seqs];
    if (h < 0 || h >= n_q_heads || t < 0 || t >= T) return -1;
    const int b = sequence_of(cu_seqlens, n_seqs, t);
    const int64_t n = t - cu_seqlens[b] + 1;
    double *z = (double *)malloc(sizeof(double) * (size_t)n);
    double *qrow = (double *)malloc(sizeof(double) * (size_t)head_dim);
    double *orow = (double *)malloc(sizeof(double) * (size_t)head_dim);
    double lse;
    if (!z || !qrow || !orow) { free(z); free(qrow); free(orow); return -1; }
    one_row(q, k, v, cu_seqlens, n_seqs, n_q_heads, n_kv_heads, head_dim, scale,
            1, T, h, t, z, qrow, orow, &lse, p_out);
    free(z); free(qrow); free(orow);
    return n;
}

/*
 * Q/K prologue, the step before attention that the h3.c README names
 * ("Profiling and diagnostic paths", "Checkpoint layout and media
 * pipeline": fused QK normalisation and rotary embedding). For every row x
 * (rows = heads * T, token t = row mod T) of a [heads][T][D] bf16 tensor:
 *   RMS norm (if w): y = x / sqrt(mean_c x_c^2 + eps) * w
 *   rotation (if tables): for i < D/2, with c = cos[t][i], s = sin[t][i],
 *     out_i       = y_i c - y_{i+D/2} s
 *     out_{i+D/2} = y_{i+D/2} c + y_i s
 * in fp64 (the caller rounds to bf16). Returns 0 on success.
 */
int oracle_qk_prep(const uint16_t *x, int64_t rows, int64_t T, int d,
                   const uint16_t *w, double eps, const float *cosv, const float *sinv,
                   double *out)
{
    if (!x || !out || rows < 0 || T <= 0 || d < 2 || (d % 2) != 0) return 1;
    if ((cosv == NULL) != (sinv == NULL)) return 2;
    const int half = d / 2;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t t = r % T;
        double *y = out + r * d;
        for (int c = 0; c < d; ++c) y[c] = bf16_bits_to_double(x[r * d + c]);
        if (w) {
            double ms = 0.0;
            for (int c = 0; c < d; ++c) ms += y[c] * y[c];
            ms /= d;
            const double inv = 1.0 / sqrt(ms + eps);
            for (int c = 0; c < d; ++c) y[c] = y[c] * inv * bf16_bits_to_double(w[c]);
        }
        if (cosv) {
            for (int i = 0; i < half; ++i) {
                const double cs = cosv[t * half + i], sn = sinv[t * half + i];
                const double a = y[i], b = y[i + half];
                y[i] = a * cs - b * sn;
                y[i + half] = b * cs + a * sn;
            }
        }
    }
    return 0;
}

/* Threads the OpenMP runtime would use (for reporting the baseline's cores). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
