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

/*
 * 8-bit KV caches.  The page "Attention over the KV cache in the decode step"
 * notes that an int8 or fp8 cache halves the bytes per cached row (and so
 * doubles the arithmetic intensity); it gives no storage format.  The reading
 * used here: every cached row of K (and of V) is d one-byte codes c[j] plus
 * one float32 scale s, and represents the values s * value(c[j]).
 *
 *   kind 1, int8      value(c) = the two's-complement integer, -128 .. 127.
 *   kind 2, fp8 e4m3  sign bit, 4 exponent bits E (bias 7), 3 mantissa bits M:
 *                     E in 1..15:  (-1)^sign * 2^(E - 7) * (1 + M / 8)
 *                     E = 0:       (-1)^sign * 2^-6 * (M / 8)   (subnormal)
 *                     E = 15, M = 7 is NaN; there are no infinities, so the
 *                     largest finite magnitude is 2^8 * 1.75 = 448.
 *
 * Quantizing a row x[0..d-1] of float32 values (absmax scaling):
 *   a = max_j |x[j]|;  s = a / Q in float32 (Q = 127 for int8, 448 for e4m3),
 *   and s = 0 when a = 0;
 *   v[j] = x[j] / s in float32, clamped to [-Q, Q] (saturation);
 *   c[j] = the code whose value is nearest v[j], ties to the even code
 *          (int8: even integer; e4m3: even mantissa), keeping the sign of a
 *          zero result; c[j] = 0 for every j when s = 0.
 * x must be finite.
 */

/* The value a code stands for (kind 1: int8, kind 2: fp8 e4m3). */
double oracle_code_value(int code, int kind)
{
    const unsigned c = (unsigned)code & 0xffu;
    if (kind == 1)
        return (double)(c >= 128 ? (int)c - 256 : (int)c);
    const int sign = (c >> 7) & 1;
    const int E = (c >> 3) & 15;
    const int M = c & 7;
    if (E == 15 && M == 7) return NAN;
    double mag;
    if (E == 0) mag = ldexp((double)M / 8.0, -6);
    else mag = ldexp(1.0 + (double)M / 8.0, E - 7);
    return sign ? -mag : mag;
}

/* Nearest e4m3 code to v (|v| <= 448), ties to the even mantissa; a zero keeps v's sign. */
static unsigned e4m3_nearest(double v)
{
    const unsigned sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x80u : 0u;
    const double a = fabs(v);  /* the caller has clamped |v| to 448 */
    /* the binade of a: spacing 2^(e-3) for normal values, 2^-9 below 2^-6 */
    int e = -6;
    if (a >= ldexp(1.0, -6)) {
        e = (int)floor(log2(a));
        /* guard against log2 rounding at exact powers of two */
        if (ldexp(1.0, e) > a) --e;
        if (ldexp(1.0, e + 1) <= a) ++e;
    }
    const double step = ldexp(1.0, e - 3);
    double q = a / step;              /* exact: a power-of-two division */
    double r = floor(q);
    const double frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    /* r counts steps of the binade: 8..16 for normal e, 0..8 for subnormal */
    int E, M;
    if (e == -6 && r < 8.0) {
        E = 0;
        M = (int)r;
    } else {
        if (r >= 16.0) {
            r = 8.0;
            ++e;
        }
        E = e + 7;
        M = (int)r - 8;
    }
    return sign | ((unsigned)E << 3) | (unsigned)M;
}

/*
 * Quantize rows x[rows][d] (float32) into codes[rows][d] and scales[rows]
 * as described above.
 */
int oracle_quantize_rows(const float *x, int64_t rows, int d, int kind,
                         uint8_t *codes, float *scales)
{
    if (!x || !codes || !scales || rows < 0 || d <= 0 || (kind != 1 && kind != 2))
        return ORACLE_ERR_ARG;
    const float Q = kind == 1 ? 127.0f : 448.0f;
    for (int64_t r = 0; r < rows; ++r) {
        const float *xr = x + r * d;
        uint8_t *cr = codes + r * d;
        float a = 0.0f;
        for (int j = 0; j < d; ++j) {
            const float m = fabsf(xr[j]);
            if (m > a) a = m;
        }
        const float s = a / Q;
        scales[r] = s;
        for (int j = 0; j < d; ++j) {
            if (s == 0.0f) {
                cr[j] = 0;
                continue;
            }
            float v = xr[j] / s;
            if (v > Q) v = Q;
            if (v < -Q) v = -Q;
            if (kind == 1) {
                const double n = nearbyint((double)v);   /* ties to even */
                cr[j] = (uint8_t)(int8_t)(int)n;
            } else {
                cr[j] = (uint8_t)e4m3_nearest((double)v);
            }
        }
    }
    return ORACLE_OK;
}

/* Values of rows of codes: out[r][j] = scales[r] * value(codes[r][j]), in double. */
int oracle_dequant_rows(const uint8_t *codes, const float *scales, int64_t rows, int d,
                        int kind, double *out)
{
    if (!codes || !scales || !out || rows < 0 || d <= 0 || (kind != 1 && kind != 2))
        return ORACLE_ERR_ARG;
    for (int64_t r = 0; r < rows; ++r)
        for (int j = 0; j < d; ++j)
            out[r * d + j] = (double)scales[r] * oracle_code_value(codes[r * d + j], kind);
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
