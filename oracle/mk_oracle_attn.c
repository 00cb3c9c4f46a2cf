/*
 * mk_oracle_attn.c -- plain, slow, fp64 CPU oracle for Ring Attention, the
 * sequence-parallel fused kernel.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code with the
 * CUDA path and neither side includes the other.
 *
 * What it computes (mKernel: Fast Multi-GPU, Multi-Node Fused Kernels,
 * Table 3, row "Ring Attention (SP)"; abstract): the sequence is cut into P
 * contiguous slices of S tokens, one per rank, and rank r holds Q_r, K_r and
 * V_r, each H heads x S rows x d columns.  Every rank's queries attend to the
 * keys and values of the whole sequence; the ring only decides the order in
 * which the other ranks' KV slices reach a rank, which moves the result by
 * rounding alone.  So for query row i of head h on rank r, over every key row
 * j of every rank o:
 *
 *     s_oj  = scale * sum_c Q_r[h][i][c] * K_o[h][j][c]
 *     m     = max over (o, j) of s_oj
 *     w_oj  = exp(s_oj - m)
 *     l     = sum over (o, j) of w_oj
 *     O_r[h][i][c] = sum over (o, j) of w_oj * V_o[h][j][c] / l
 *     lse_r[h][i]  = m + log(l)                    (natural-log logsumexp)
 *
 * This is softmax attention written out; subtracting the maximum changes
 * nothing mathematically and keeps exp() finite.
 *
 * Arithmetic: bf16 inputs are widened exactly to fp64; every sum runs in
 * increasing index order (ranks o = 0..P-1, then rows j, then columns c) in
 * fp64; exp and log are the C library's.  No blocking, no reordering, no
 * fused multiply-add (the build passes -ffp-contract=off).
 *
 * Besides O and lse, the oracle returns for every output element
 *     e[i][c] = sqrt(sum over (o, j) of w_oj^2 * V_o[h][j][c]^2) / l,
 * the scale of the error that rounding each probability w_oj / l (relative)
 * to a narrower format adds to O[i][c]: with independent relative rounding
 * errors of standard deviation u, that error has standard deviation u * e.
 * The GPU tests derive their tolerance from it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Query rows rows[0..n) of head `head` on rank `rank`.  Q, K, V are arrays of
 * P pointers to H x S x d bf16 tensors (row-major).  Outputs: O and err are
 * n x d, lse is n (fp64).
 */
void mko_attention_rows(int P, int64_t H, int64_t S, int64_t d, const uint16_t *const *Q,
                        const uint16_t *const *K, const uint16_t *const *V, int rank, int64_t head,
                        int64_t n, const int64_t *rows, double scale, double *O, double *lse,
                        double *err) {
    (void)H;
    const int64_t nkeys = (int64_t)P * S;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(nkeys > 0 ? nkeys : 1));
        double *q = (double *)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
        double *acc = (double *)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
        double *acc2 = (double *)malloc(sizeof(double) * (size_t)(d > 0 ? d : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t t = 0; t < n; ++t) {
            const uint16_t *qrow = Q[rank] + (head * S + rows[t]) * d;
            for (int64_t c = 0; c < d; ++c) q[c] = bf16_value(qrow[c]);
            /* scores over every key, ranks in order */
            double m = -INFINITY;
            for (int o = 0; o < P; ++o) {
                for (int64_t j = 0; j < S; ++j) {
                    const uint16_t *krow = K[o] + (head * S + j) * d;
                    double dot = 0.0;
                    for (int64_t c = 0; c < d; ++c) dot += q[c] * bf16_value(krow[c]);
                    const double sc = scale * dot;
                    s[(int64_t)o * S + j] = sc;
                    if (sc > m) m = sc;
                }
            }
            double l = 0.0;
            for (int64_t c = 0; c < d; ++c) acc[c] = acc2[c] = 0.0;
            for (int o = 0; o < P; ++o) {
                for (int64_t j = 0; j < S; ++j) {
                    const double w = exp(s[(int64_t)o * S + j] - m);
                    l += w;
                    const uint16_t *vrow = V[o] + (head * S + j) * d;
                    for (int64_t c = 0; c < d; ++c) {
                        const double v = bf16_value(vrow[c]);
                        acc[c] += w * v;
                        acc2[c] += (w * v) * (w * v);
                    }
                }
            }
            for (int64_t c = 0; c < d; ++c) {
                O[t * d + c] = acc[c] / l;
                err[t * d + c] = sqrt(acc2[c]) / l;
            }
            lse[t] = m + log(l);
        }
        free(s);
        free(q);
        free(acc);
        free(acc2);
    }
}
