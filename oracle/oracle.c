/*
 * oracle.c -- arithmetic core of the CPU oracle for the sharded matmul
 * A[I,J] . B[J,K] -> C[I,K] with partial-sum reduction.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header or constant with the CUDA path and must never be used to produce
 * a product result.
 *
 * Every routine is the plain definition of one step of the method:
 *   - the per-rank local product ("each rank computes C_r over its slice of
 *     the contracted dimension", Sharded matrix multiplication and result
 *     ownership, steps 2-3; Row Parallelism, partial result Z_i = X_i A_i);
 *   - the sum of the partials "with matching output coordinates" (same page,
 *     step 4; Row Parallelism, Y = sum_i X_i A_i), in ascending rank order in
 *     fp32, or as a balanced pairwise tree for the tree variant;
 *   - rounding to the stored element size (bfloat16, round to nearest even);
 *   - the GeLU activation between the two MLP matmuls (The simple maths
 *     behind parallel training, "MLP block"), tanh form.
 * Floating point: products are accumulated in double and the partial is
 * stored as fp32, mirroring an fp32 partial-sum buffer.  Compile with
 * -ffp-contract=off so no multiply-add is fused on any host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- bfloat16 rounding ------------------------------------------------ */

/* bfloat16 keeps the sign, the 8 exponent bits and the 7 leading fraction
 * bits of an IEEE binary32 value: it is the upper half of the binary32 bit
 * pattern.  Round to nearest, ties to even, on the discarded lower 16 bits.
 * NaN stays NaN (quiet); infinities pass through; overflow rounds to inf. */
float orc_round_bf16(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    if ((u & 0x7f800000u) == 0x7f800000u) {
        if (u & 0x007fffffu)
            u |= 0x00400000u; /* NaN: force the quiet bit, which survives */
        u &= 0xffff0000u;
    } else {
        uint32_t lower = u & 0x0000ffffu;
        uint32_t upper = u >> 16;
        /* lower > half, or exactly half with an odd kept part: round up */
        if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u)))
            upper += 1u; /* a carry into the exponent is the correct result */
        u = upper << 16;
    }
    memcpy(&x, &u, sizeof x);
    return x;
}

void orc_round_bf16_array(const float *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_round_bf16(in[i]);
}

/* ---- local product of one rank ---------------------------------------- */

/* P[i][k] = fp32( sum_{j=0}^{J-1} A[row_i][j] * B[j][k] ), the sum taken in
 * double in ascending j.  A is row-major with leading dimension lda, B with
 * ldb, P with ldp.  rows == NULL means row_i = i for i < nrows; otherwise
 * only the listed rows of A are formed (sampled outputs), P row i holding
 * A row rows[i].  nthreads > 1 splits the output rows across threads; every
 * output element is still one sequential sum. */
void orc_local_product(const float *A, int64_t lda, const float *B, int64_t ldb,
                       float *P, int64_t ldp, int64_t nrows, const int64_t *rows,
                       int64_t J, int64_t K, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t i = 0; i < nrows; ++i) {
        const float *a = A + (rows ? rows[i] : i) * lda;
        double *acc = (double *)calloc((size_t)(K > 0 ? K : 1), sizeof(double));
        for (int64_t j = 0; j < J; ++j) {
            const double aij = (double)a[j];
            const float *b = B + j * ldb;
            for (int64_t k = 0; k < K; ++k)
                acc[k] += aij * (double)b[k];
        }
        float *p = P + i * ldp;
        for (int64_t k = 0; k < K; ++k)
            p[k] = (float)acc[k];
        free(acc);
    }
}

/* Dense product in double, no rounding: D[i][k] = sum_j A[i][j] * B[j][k].
 * Used only to check the identity "sum of the partials = dense product". */
void orc_dense_product_f64(const double *A, const double *B, double *D,
                           int64_t I, int64_t J, int64_t K)
{
    for (int64_t i = 0; i < I; ++i) {
        double *d = D + i * K;
        for (int64_t k = 0; k < K; ++k)
            d[k] = 0.0;
        for (int64_t j = 0; j < J; ++j) {
            const double aij = A[i * J + j];
            const double *b = B + j * K;
            for (int64_t k = 0; k < K; ++k)
                d[k] += aij * b[k];
        }
    }
}

/* ---- sum of the partials over the ranks of one reduction group -------- */

/* out[e] = ((parts[0][e] + parts[1][e]) + parts[2][e]) + ... in fp32, the
 * canonical order: ascending rank id, one fp32 rounding per addition. */
void orc_sum_sequential(const float *const *parts, int n, int64_t len, float *out)
{
    for (int64_t e = 0; e < len; ++e) {
        float s = parts[0][e];
        for (int r = 1; r < n; ++r)
            s = s + parts[r][e];
        out[e] = s;
    }
}

/* Balanced pairwise tree over the ranks in ascending order: the leaves are
 * parts[0..n-1], padded with -0.0 (the additive identity for every fp32
 * value, signed zeros included) up to the next power of two; each inner
 * node is the fp32 sum of its left and right child. */
void orc_sum_pairwise(const float *const *parts, int n, int64_t len, float *out)
{
    int width = 1;
    while (width < n)
        width <<= 1;
    float *level = (float *)malloc((size_t)width * sizeof(float));
    const float neg_zero = -0.0f;
    for (int64_t e = 0; e < len; ++e) {
        for (int r = 0; r < width; ++r)
            level[r] = (r < n) ? parts[r][e] : neg_zero;
        for (int w = width; w > 1; w >>= 1)
            for (int r = 0; r < w / 2; ++r)
                level[r] = level[2 * r] + level[2 * r + 1];
        out[e] = level[0];
    }
    free(level);
}

/* ---- GeLU ----------------------------------------------------------- */

/* GeLU, tanh form (Hendrycks & Gimpel, 2016):
 *   gelu(x) = x/2 * (1 + tanh( sqrt(2/pi) * (x + 0.044715 x^3) ))
 * evaluated in double. */
double orc_gelu_tanh(double x)
{
    const double c = sqrt(2.0 / 3.14159265358979323846);
    return 0.5 * x * (1.0 + tanh(c * (x + 0.044715 * x * x * x)));
}

void orc_gelu_tanh_array(const float *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)orc_gelu_tanh((double)in[i]);
}
