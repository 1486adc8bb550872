/*
 * Plain CPU oracle for decode-step attention over a KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA path is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * product library never links or calls it, and it shares no code, header or
 * table with the CUDA sources.
 *
 * Arithmetic is IEEE double throughout.  Inputs arrive as float32 arrays
 * (a bf16 cache is widened to float32 by the caller, which is exact), so the
 * oracle sees exactly the rounded values the GPU reads.
 *
 * Source of each step ("MoA-Structured Decode Attention", arXiv 2607.19456):
 *   - Step I   (section 2, eq. 1): s[l] = scale * sum_j q[j] * K[l][j],
 *              K read row by row in its natural row-major layout.
 *   - Step II  (section 2, eq. 2): m = max_l s[l]; e[l] = exp(s[l] - m);
 *              Z = sum_l e[l]; a[l] = e[l] / Z.
 *   - Step III (section 2, eq. 3): out[d] = sum_l a[l] * V[l][d].
 *   - Row-major gamma offsets (section 3): element <l, j> of a rank-2 K lives
 *              at l * d_k + j; the rank-4 cache <B, h_kv, n_max, d_k> lifts
 *              this to ((b * h_kv + h) * n_max + l) * d_k + j.
 *   - KV accumulation '#' (introduction, item 3): one new row is written
 *              per head at its precomputed gamma offset.
 *   - GQA/MQA psi-selection (introduction, item 4): query head h reads KV
 *              head h / (h_q / h_kv); the broadcast is never materialised.
 *   - Full causal attention (page "StoryLM-0 head-parallel attention",
 *              section 3): softmax(scale * Q K^T + mask) V with a
 *              strictly-upper-triangular -inf mask, used only as a
 *              cross-check of the decode definition.
 *
 * The three steps are written as three separate passes over the cached rows
 * with explicit buffers for s and a; there is no online softmax, no blocking
 * and no splitting here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Return codes. */
#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_NOMEM (-2)

/*
 * One head, one query row, n cached rows (section 2, Steps I-III).
 *   q   : [d_k]
 *   K   : [n][d_k] row-major (row stride d_k)
 *   V   : [n][d_v] row-major (row stride d_v)
 *   out : [d_v]            written
 *   a   : [n] or NULL      softmax weights, written when non-NULL
 *   lse : scalar or NULL   m + log(Z), the log of the softmax denominator
 *                          taken on the scaled scores; -INFINITY when n == 0
 * With n == 0 the softmax is over an empty set; the oracle defines out = 0
 * and lse = -inf for it (the pages do not cover this case).
 */
int oracle_decode_head(const float *q, const float *K, const float *V,
                       int64_t n, int d_k, int d_v, double scale,
                       double *out, double *a, double *lse)
{
    if (!q || !out || d_k <= 0 || d_v <= 0 || n < 0) return ORACLE_ERR_ARG;
    if (n > 0 && (!K || !V)) return ORACLE_ERR_ARG;

    if (n == 0) {
        for (int d = 0; d < d_v; ++d) out[d] = 0.0;
        if (lse) *lse = -INFINITY;
        return ORACLE_OK;
    }

    double *s = (double *)malloc((size_t)n * sizeof(double));
    double *w = (double *)malloc((size_t)n * sizeof(double));
    if (!s || !w) { free(s); free(w); return ORACLE_ERR_NOMEM; }

    /* Step I: scores, one inner product per cached row of K. */
    for (int64_t l = 0; l < n; ++l) {
        double acc = 0.0;
        for (int j = 0; j < d_k; ++j)
            acc += (double)q[j] * (double)K[l * d_k + j];
        s[l] = scale * acc;
    }

    /* Step II: numerically stable softmax over the score vector. */
    double m = s[0];
    for (int64_t l = 1; l < n; ++l)
        if (s[l] > m) m = s[l];
    double Z = 0.0;
    for (int64_t l = 0; l < n; ++l) {
        w[l] = exp(s[l] - m);
        Z += w[l];
    }
    for (int64_t l = 0; l < n; ++l) w[l] = w[l] / Z;

    /* Step III: weighted sum of the rows of V. */
    for (int d = 0; d < d_v; ++d) {
        double acc = 0.0;
        for (int64_t l = 0; l < n; ++l)
            acc += w[l] * (double)V[l * d_v + d];
        out[d] = acc;
    }

    if (a) memcpy(a, w, (size_t)n * sizeof(double));
    if (lse) *lse = m + log(Z);
    free(s);
    free(w);
    return ORACLE_OK;
}

/*
 * Batched, multi-head decode over a padded cache (section 2 lifted by the
 * Omega rank argument; GQA psi-selection from the introduction, item 4).
 *   q        : [B][h_q][d_k]
 *   K        : [B][h_kv][n_max][d_k]
 *   V        : [B][h_kv][n_max][d_v]
 *   seq_lens : [B], 0 <= seq_lens[b] <= n_max (rows 0..seq_lens[b]-1 are read)
 *   out      : [B][h_q][d_v]   written
 *   lse      : [B][h_q] or NULL
 *   threads  : OpenMP threads over the independent (b, h) pairs (>= 1)
 */
int oracle_decode(const float *q, const float *K, const float *V,
                  const int32_t *seq_lens, double *out, double *lse,
                  int B, int h_q, int h_kv, int d_k, int d_v, int64_t n_max,
                  double scale, int threads)
{
    if (!q || !K || !V || !seq_lens || !out) return ORACLE_ERR_ARG;
    if (B <= 0 || h_q <= 0 || h_kv <= 0 || d_k <= 0 || d_v <= 0 || n_max < 0)
        return ORACLE_ERR_ARG;
    if (h_q % h_kv != 0) return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > n_max) return ORACLE_ERR_ARG;
    if (threads < 1) threads = 1;

    const int group = h_q / h_kv;
    int status = ORACLE_OK;
    const int64_t units = (int64_t)B * h_q;

#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
    for (int64_t u = 0; u < units; ++u) {
        const int b = (int)(u / h_q);
        const int h = (int)(u % h_q);
        const int kvh = h / group;
        const int64_t row0 = ((int64_t)b * h_kv + kvh) * n_max;
        int rc = oracle_decode_head(q + u * d_k, K + row0 * d_k, V + row0 * d_v,
                                    seq_lens[b], d_k, d_v, scale,
                                    out + u * d_v, NULL, lse ? lse + u : NULL);
        if (rc != ORACLE_OK) {
#pragma omp critical
            status = rc;
        }
    }
    return status;
}

/*
 * Log-sum-exp merge of partial results over disjoint row ranges.  Each part
 * s carries the normalised output o_s (the decode of its own rows) and its
 * lse_s = m_s + log(Z_s).  Over the union the softmax denominator is
 * Z = sum_s exp(lse_s), so part s holds the fraction exp(lse_s) / Z of the
 * total weight and out = sum_s (exp(lse_s) / Z) * o_s.  Written with the
 * largest lse subtracted first, as in Step II.  Parts with lse = -inf hold
 * no rows and get weight 0; if every part is empty out = 0 and lse = -inf.
 *   o_parts : [S][d_v]   lse_parts : [S]   out : [d_v]   lse : scalar or NULL
 */
int oracle_lse_combine(const double *o_parts, const double *lse_parts, int S,
                       int d_v, double *out, double *lse)
{
    if (!o_parts || !lse_parts || !out || S < 0 || d_v <= 0)
        return ORACLE_ERR_ARG;
    double L = -INFINITY;
    for (int s = 0; s < S; ++s)
        if (lse_parts[s] > L) L = lse_parts[s];
    if (L == -INFINITY) {
        for (int d = 0; d < d_v; ++d) out[d] = 0.0;
        if (lse) *lse = -INFINITY;
        return ORACLE_OK;
    }
    double Z = 0.0;
    for (int s = 0; s < S; ++s) Z += exp(lse_parts[s] - L);
    for (int d = 0; d < d_v; ++d) {
        double acc = 0.0;
        for (int s = 0; s < S; ++s)
            acc += (exp(lse_parts[s] - L) / Z) * o_parts[(int64_t)s * d_v + d];
        out[d] = acc;
    }
    if (lse) *lse = L + log(Z);
    return ORACLE_OK;
}

/*
 * KV-cache accumulation (introduction, item 3; gamma offsets of section 3):
 * for every (b, h) copy the new key row k_new[b][h][:] into
 * K[b][h][pos[b]][:] and the new value row into V likewise, byte for byte.
 * Rows whose pos[b] lies outside [0, n_max) are not written; the return
 * value is the number of such sequences (0 when every row was written).
 *   elem_size : bytes per element (4 for fp32, 2 for bf16); the copy is
 *               exact whatever the element type.
 */
int oracle_kv_append(const void *k_new, const void *v_new, void *K, void *V,
                     const int32_t *pos, int B, int h_kv, int d_k, int d_v,
                     int64_t n_max, int elem_size)
{
    if (!k_new || !v_new || !K || !V || !pos) return ORACLE_ERR_ARG;
    if (B <= 0 || h_kv <= 0 || d_k <= 0 || d_v <= 0 || n_max <= 0 || elem_size <= 0)
        return ORACLE_ERR_ARG;
    int skipped = 0;
    for (int b = 0; b < B; ++b) {
        const int64_t p = pos[b];
        if (p < 0 || p >= n_max) { ++skipped; continue; }
        for (int h = 0; h < h_kv; ++h) {
            const int64_t row = ((int64_t)b * h_kv + h) * n_max + p;
            const int64_t src = (int64_t)b * h_kv + h;
            memcpy((char *)K + row * d_k * elem_size,
                   (const char *)k_new + src * d_k * elem_size,
                   (size_t)d_k * elem_size);
            memcpy((char *)V + row * d_v * elem_size,
                   (const char *)v_new + src * d_v * elem_size,
                   (size_t)d_v * elem_size);
        }
    }
    return skipped;
}

/*
 * Full causal attention for H heads over T tokens ("StoryLM-0 head-parallel
 * attention", section 3): for each head, the whole T x T score matrix
 * scale * Q K^T, an additive mask of -inf above the diagonal, a row softmax,
 * and the product with V.  This is the prefill form; its last row is what a
 * decode step over T cached rows must reproduce.
 *   Q : [H][T][d_k]   K : [H][T][d_k]   V : [H][T][d_v]   out : [H][T][d_v]
 */
int oracle_causal_attention(const float *Q, const float *K, const float *V,
                            int H, int T, int d_k, int d_v, double scale,
                            double *out)
{
    if (!Q || !K || !V || !out || H <= 0 || T <= 0 || d_k <= 0 || d_v <= 0)
        return ORACLE_ERR_ARG;
    double *S = (double *)malloc((size_t)T * T * sizeof(double));
    if (!S) return ORACLE_ERR_NOMEM;
    for (int h = 0; h < H; ++h) {
        const float *Qh = Q + (int64_t)h * T * d_k;
        const float *Kh = K + (int64_t)h * T * d_k;
        const float *Vh = V + (int64_t)h * T * d_v;
        double *Oh = out + (int64_t)h * T * d_v;
        /* scores plus mask */
        for (int i = 0; i < T; ++i)
            for (int j = 0; j < T; ++j) {
                double acc = 0.0;
                for (int c = 0; c < d_k; ++c)
                    acc += (double)Qh[i * d_k + c] * (double)Kh[j * d_k + c];
                S[i * T + j] = (j > i) ? -INFINITY : scale * acc;
            }
        /* row softmax */
        for (int i = 0; i < T; ++i) {
            double m = -INFINITY;
            for (int j = 0; j < T; ++j)
                if (S[i * T + j] > m) m = S[i * T + j];
            double Z = 0.0;
            for (int j = 0; j < T; ++j) {
                S[i * T + j] = exp(S[i * T + j] - m);
                Z += S[i * T + j];
            }
            for (int j = 0; j < T; ++j) S[i * T + j] /= Z;
        }
        /* probabilities times V */
        for (int i = 0; i < T; ++i)
            for (int d = 0; d < d_v; ++d) {
                double acc = 0.0;
                for (int j = 0; j < T; ++j)
                    acc += S[i * T + j] * (double)Vh[j * d_v + d];
                Oh[i * d_v + d] = acc;
            }
    }
    free(S);
    return ORACLE_OK;
}

/* Number of OpenMP threads a parallel region may use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
