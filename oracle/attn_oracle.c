/*
 * Exact-attention oracle: plain, slow, fp64 CPU reference.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * What it computes is the plain definition of scaled dot-product attention
 * ("6.1 FlashAttention V1 in detail", section 1.1: S = Q K^T / sqrt(d),
 * P = softmax(S), O = P V), with the softmax taken literally as the three-pass
 * safe softmax of the same page, section 3.1 (pass 1: row max; pass 2: sum of
 * exp(x - max); pass 3: exp(x - max) / sum), and the per-row log-sum-exp that
 * "FlashAttention: IO-Aware Tiling, Online Softmax Mathematics, ..." (section
 * "Backward Pass Recomputation") stores as L = m + log(l).
 *
 * Readings where the pages are silent:
 *   - the scale is an argument (the configs use 1/sqrt(d)); it is applied to
 *     the dot product exactly as given, in double;
 *   - causal masking keeps keys j <= i for query row i (square problem, so
 *     top-left and bottom-right alignment coincide); masked keys take no part
 *     in the max, the sum or the output;
 *   - the log is the natural log, over the scaled logits.
 *
 * Inputs are bf16 bit patterns, widened exactly to double, so the oracle sees
 * the very values the GPU sees.  All arithmetic is double; no fast-math.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One query row i of one (batch, head) slice, over the admitted keys j with
 * kv_lo <= j < kv_hi (and j <= i when causal).
 *   qh, kh, vh : the slice's [N, d] row-major bf16 matrices
 *   s          : caller scratch of N doubles (the row of S)
 *   o_row      : d doubles out
 *   lse        : one double out
 * A row that admits no key gets O = 0 and LSE = -inf (it carries no weight
 * when partial results over disjoint key ranges are merged).
 */
static void oracle_row(const uint16_t *qh, const uint16_t *kh, const uint16_t *vh,
                       int64_t N, int64_t d, double scale, int causal, int64_t i,
                       int64_t kv_lo, int64_t kv_hi, double *s, double *o_row, double *lse)
{
    int64_t j_end = causal ? (i + 1) : N; /* keys admitted to row i: [kv_lo, j_end) */
    if (j_end > kv_hi) j_end = kv_hi;
    const uint16_t *q = qh + i * d;

    for (int64_t c = 0; c < d; ++c) o_row[c] = 0.0;
    if (j_end <= kv_lo) {
        *lse = -INFINITY;
        return;
    }

    /* S_ij = scale * sum_c Q_ic K_jc */
    for (int64_t j = kv_lo; j < j_end; ++j) {
        const uint16_t *kr = kh + j * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c)
            acc += widen_bf16(q[c]) * widen_bf16(kr[c]);
        s[j] = scale * acc;
    }

    /* pass 1: m = max_j S_ij */
    double m = -INFINITY;
    for (int64_t j = kv_lo; j < j_end; ++j)
        if (s[j] > m) m = s[j];

    /* pass 2: l = sum_j exp(S_ij - m) */
    double l = 0.0;
    for (int64_t j = kv_lo; j < j_end; ++j)
        l += exp(s[j] - m);

    /* pass 3: P_ij = exp(S_ij - m) / l, then O_i = sum_j P_ij V_j */
    for (int64_t j = kv_lo; j < j_end; ++j) {
        const double p = exp(s[j] - m) / l;
        const uint16_t *vr = vh + j * d;
        for (int64_t c = 0; c < d; ++c)
            o_row[c] += p * widen_bf16(vr[c]);
    }

    *lse = m + log(l);
}

/*
 * Attention over a set of rows.
 *
 *   q, k, v  : bf16 bits, contiguous [B, H, N, d]
 *   rows     : flat row ids r = (b*H + h)*N + i, n_rows of them; NULL means
 *              every row in order (n_rows must then be B*H*N)
 *   o        : n_rows * d doubles out, row-major in the order of `rows`
 *   lse      : n_rows doubles out
 *   threads  : worker threads (<= 0: the OpenMP default)
 *   kv_lo, kv_hi : only keys kv_lo <= j < kv_hi take part (0, N: all keys)
 *
 * Returns 0, or -1 on an invalid argument (nothing written).
 */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                          int64_t B, int64_t H, int64_t N, int64_t d,
                          double scale, int causal,
                          const int64_t *rows, int64_t n_rows,
                          double *o, double *lse, int threads,
                          int64_t kv_lo, int64_t kv_hi)
{
    if (!q || !k || !v || !o || !lse || B < 1 || H < 1 || N < 1 || d < 1 || n_rows < 0)
        return -1;
    if (kv_lo < 0 || kv_hi > N || kv_lo >= kv_hi)
        return -1;
    if (!rows && n_rows != B * H * N)
        return -1;
    if (rows) {
        for (int64_t t = 0; t < n_rows; ++t)
            if (rows[t] < 0 || rows[t] >= B * H * N) return -1;
    }
    int failed = 0;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t t = 0; t < n_rows; ++t) {
            if (!s) continue;
            const int64_t r = rows ? rows[t] : t;
            const int64_t bh = r / N, i = r % N;
            const int64_t base = bh * N * d;
            oracle_row(q + base, k + base, v + base, N, d, scale, causal, i, kv_lo, kv_hi, s,
                       o + t * d, lse + t);
        }
        free(s);
    }
    return failed ? -2 : 0;
}

/* Threads the library would use by default (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
