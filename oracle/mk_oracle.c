/*
 * mk_oracle.c -- plain, slow, fp64 CPU oracle for the rank-summed GEMM of
 * row-parallel tensor parallelism (GEMM + AllReduce / GEMM + ReduceScatter /
 * AllGather + GEMM).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code with the
 * CUDA path and neither side includes the other.
 *
 * What it computes (mKernel: Fast Multi-GPU, Multi-Node Fused Kernels,
 * Table 3, rows "GEMM + AllReduce (TP)" and "GEMM + ReduceScatter (TP)"):
 * with the K dimension split over P ranks, rank r holds A_r (M x K_r) and
 * B_r (K_r x N); the collective sums the per-rank products, so
 *
 *     C[i][j] = sum_{r=0}^{P-1} p_r[i][j],   p_r[i][j] = sum_{k=0}^{K_r-1} A_r[i][k] B_r[k][j].
 *
 * Arithmetic: every bf16 input is widened exactly to fp64; each p_r element
 * is accumulated in fp64 over k in increasing order; the rank sum runs over r
 * in increasing order.  No blocking, no reordering, no fused multiply-add
 * (the build passes -ffp-contract=off).  Output rounding to bf16 is
 * round-to-nearest-even applied directly to the fp64 value (no detour
 * through fp32, so there is no double rounding).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 bit pattern -> exact fp64 value (bf16 is the top half of an fp32). */
static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Rows [i0, i0+ni) of one dense product X * Y, X m x k row-major, Y k x n
 * row-major, both bf16 bits; out is ni x n doubles.
 * out[i][j] = sum over kk = 0..k-1 (increasing) of X[i][kk] * Y[kk][j].
 */
void mko_gemm_rows(int64_t n, int64_t k, const uint16_t *X, const uint16_t *Y,
                   int64_t i0, int64_t ni, double *out) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ii = 0; ii < ni; ++ii) {
        const int64_t i = i0 + ii;
        double *o = out + ii * n;
        for (int64_t j = 0; j < n; ++j) o[j] = 0.0;
        for (int64_t kk = 0; kk < k; ++kk) {
            const double x = bf16_value(X[i * k + kk]);
            const uint16_t *y = Y + kk * n;
            for (int64_t j = 0; j < n; ++j) o[j] += x * bf16_value(y[j]);
        }
    }
}

/*
 * Rows [i0, i0+ni) of C = sum_r A_r B_r (the AllReduce result): for each row,
 * p_r is formed in full in fp64 and added to the running sum in rank order
 * r = 0, 1, ..., P-1.
 */
void mko_rank_sum_rows(int P, int64_t N, int64_t Kr, const uint16_t *const *A,
                       const uint16_t *const *B, int64_t i0, int64_t ni, double *C) {
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t ii = 0; ii < ni; ++ii) {
            const int64_t i = i0 + ii;
            double *c = C + ii * N;
            for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
            for (int r = 0; r < P; ++r) {
                for (int64_t j = 0; j < N; ++j) p[j] = 0.0;
                for (int64_t kk = 0; kk < Kr; ++kk) {
                    const double a = bf16_value(A[r][i * Kr + kk]);
                    const uint16_t *b = B[r] + kk * N;
                    for (int64_t j = 0; j < N; ++j) p[j] += a * bf16_value(b[j]);
                }
                for (int64_t j = 0; j < N; ++j) c[j] += p[j];
            }
        }
        free(p);
    }
}

/*
 * The same sum at ns chosen elements (rows[s], cols[s]), in the same order of
 * operations as mko_rank_sum_rows, so both give identical fp64 values.
 */
void mko_rank_sum_at(int P, int64_t N, int64_t Kr, const uint16_t *const *A,
                     const uint16_t *const *B, int64_t ns, const int64_t *rows,
                     const int64_t *cols, double *out) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t s = 0; s < ns; ++s) {
        const int64_t i = rows[s], j = cols[s];
        double c = 0.0;
        for (int r = 0; r < P; ++r) {
            double p = 0.0;
            for (int64_t kk = 0; kk < Kr; ++kk)
                p += bf16_value(A[r][i * Kr + kk]) * bf16_value(B[r][kk * N + j]);
            c += p;
        }
        out[s] = c;
    }
}

/*
 * fp64 -> bf16 bits, round to nearest, ties to even, straight from fp64.
 * bf16 keeps 8 significant bits; normal exponents span [-126, 127] and the
 * subnormal quantum is 2^-133.  Magnitudes that round above the largest
 * finite bf16 become infinity; NaN becomes the quiet NaN 0x7FC0.
 */
static uint16_t round_bf16_one(double x) {
    if (isnan(x)) return 0x7FC0u;
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    const double ax = fabs(x);
    if (isinf(ax)) return sign | 0x7F80u;
    if (ax == 0.0) return sign;
    int e;
    (void)frexp(ax, &e);           /* ax = m * 2^e, m in [0.5, 1): leading bit is 2^(e-1) */
    int lead = e - 1;
    if (lead < -126) lead = -126;  /* subnormal range: fixed quantum */
    const double quantum = ldexp(1.0, lead - 7);
    const double q = nearbyint(ax / quantum); /* exact scaling; default mode is nearest-even */
    const double y = q * quantum;
    const double max_finite = ldexp(255.0, 127 - 7); /* (2 - 2^-7) * 2^127 */
    if (y > max_finite) return sign | 0x7F80u;
    const float f = (float)y;      /* exact: y has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFFu);
}

void mko_round_bf16(const double *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_bf16_one(x[i]);
}

/* fp64 -> fp32, round to nearest even (the C conversion in the default mode). */
void mko_round_f32(const double *x, int64_t n, float *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (float)x[i];
}
