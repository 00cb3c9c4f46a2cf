/*
 * Seeded synthetic input generator shared by the tests, the bench and the
 * oracle's callers.  It produces bf16 bit patterns only; it holds none of the
 * arithmetic of the rank-summed GEMM itself.
 *
 * Random bits: Philox4x32-10, the counter-based generator of Salmon, Moraes,
 * Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11):
 * ten rounds of two 32x32->64 multiplies with the published multipliers,
 * a Weyl-sequence key schedule between rounds.
 *
 * Stream layout (one independent stream per tensor of every logical rank):
 *   key     = (seed, rank)
 *   counter = (block index low 32 bits, block index high 32 bits, tensor id, 0)
 *   element e uses word e % 4 of block e / 4.
 *
 * Value recipes (all rounded to bf16 with round-to-nearest-even through fp32):
 *   DIST_UNIFORM : lo + (hi - lo) * u,  u = (w >> 8) * 2^-24 in [0, 1)
 *   DIST_NORMAL  : mean + sqrt(var) * z, z from the Box-Muller transform of
 *                  two such uniforms (the radius uses 1 - u so log() never sees 0);
 *                  one block of four words gives four normals
 *   DIST_INTEGER : lo + floor(u * (hi - lo + 1)), integers in [lo, hi]
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void ig_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += PHILOX_W0;
        k1 += PHILOX_W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* fp32 -> bf16 bits, round to nearest even (NaN kept quiet). */
static uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static double unit_u24(uint32_t w) { return (double)(w >> 8) * (1.0 / 16777216.0); }

enum { DIST_UNIFORM = 0, DIST_NORMAL = 1, DIST_INTEGER = 2 };

/* Fill out[0..n) with the elements [first, first + n) of the stream
 * (seed, rank, tensor_id).  Returns 0, or -1 for an unknown distribution. */
int ig_fill_bf16(uint16_t *out, int64_t first, int64_t n, int dist, double p0, double p1,
                 uint32_t seed, uint32_t rank, uint32_t tensor_id) {
    if (dist < 0 || dist > 2) return -1;
    if (n <= 0) return 0;
    const double two_pi = 6.283185307179586476925286766559;
    const int64_t b_first = first / 4;
    const int64_t b_last = (first + n - 1) / 4;
#pragma omp parallel for schedule(static)
    for (int64_t b = b_first; b <= b_last; ++b) {
        uint32_t ctr[4] = {(uint32_t)(uint64_t)b, (uint32_t)((uint64_t)b >> 32), tensor_id, 0u};
        uint32_t key[2] = {seed, rank};
        uint32_t w[4];
        ig_philox4x32_10(ctr, key, w);
        double v[4];
        if (dist == DIST_UNIFORM) {
            for (int q = 0; q < 4; ++q) v[q] = p0 + (p1 - p0) * unit_u24(w[q]);
        } else if (dist == DIST_INTEGER) {
            double span = p1 - p0 + 1.0;
            for (int q = 0; q < 4; ++q) v[q] = p0 + floor(unit_u24(w[q]) * span);
        } else {
            double sd = sqrt(p1);
            for (int pair = 0; pair < 2; ++pair) {
                double u1 = 1.0 - unit_u24(w[2 * pair]); /* (0, 1] */
                double u2 = unit_u24(w[2 * pair + 1]);
                double rad = sqrt(-2.0 * log(u1));
                v[2 * pair] = p0 + sd * rad * cos(two_pi * u2);
                v[2 * pair + 1] = p0 + sd * rad * sin(two_pi * u2);
            }
        }
        for (int q = 0; q < 4; ++q) {
            int64_t e = b * 4 + q;
            if (e < first || e >= first + n) continue;
            out[e - first] = f32_to_bf16_bits((float)v[q]);
        }
    }
    return 0;
}
