/*
 * grgen.c -- seeded, counter-based generator of synthetic inputs (weights,
 * prompt tokens, pre-filled KV, page permutations).
 *
 * This module is shared by the tests, the benchmark and the oracle's callers.
 * It holds none of the decode step's arithmetic: it only turns
 * (seed, stream, index) into numbers.
 *
 * Definition (platform independent: integer work plus IEEE-754 +,-,*,/ in a
 * fixed order, built with -ffp-contract=off; no libm transcendental calls):
 *
 *   word(seed, stream, i) = mix(key + (i + 1) * GAMMA)
 *   key(seed, stream)     = mix(mix(seed + GAMMA) ^ (stream * GAMMA2))
 *   mix                   = the splitmix64 output function (Steele, Lea and
 *                           Flood, "Fast splittable pseudorandom number
 *                           generators", OOPSLA 2014; constants of Vigna's
 *                           public-domain splitmix64).
 *
 *   normal(i) = mean + sigma * Z[word >> 48], where Z is a 65536-entry table
 *   of standard-normal quantiles at the cell midpoints (k + 0.5) / 65536,
 *   solved by Newton's method on the normal CDF (series expansion, own exp).
 *   The distribution is N(mean, sigma^2) quantised to 65536 levels and
 *   truncated at +-4.33 sigma.
 *
 *   uniform int in [lo, hi): lo + ((word >> 32) * (hi - lo)) >> 32
 *   (Lemire's multiply-shift; bias < 2^-32 * (hi - lo)).
 *
 *   permutation(n): Fisher-Yates, swap i with uniform[0, i] drawn from word(i).
 */
#include <stdint.h>
#include <string.h>

#define GAMMA  0x9E3779B97F4A7C15ULL
#define GAMMA2 0xD1B54A32D192ED03ULL
#define NQ 65536

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GAMMA) ^ (stream * GAMMA2));
}

uint64_t grgen_word(uint64_t seed, uint64_t stream, uint64_t i) {
    return mix64(stream_key(seed, stream) + (i + 1) * GAMMA);
}

/* ---- deterministic exp and normal CDF (no libm) ---- */

/* 2^k for integer k in the normal range, built from the exponent field. */
static double pow2i(int k) {
    uint64_t bits = (uint64_t)(k + 1023) << 52;
    double r;
    memcpy(&r, &bits, sizeof r);
    return r;
}

/* exp(x) for x in [-800, 0]: Cody-Waite reduction x = k ln2 + r, |r| <= ln2/2,
   then a 24-term Taylor series; deterministic, not correctly rounded. */
static double det_exp(double x) {
    const double LN2_HI = 6.93147180369123816490e-01;
    const double LN2_LO = 1.90821492927058770002e-10;
    const double INV_LN2 = 1.44269504088896338700e+00;
    if (x < -700.0) return 0.0;
    double t = x * INV_LN2;
    int k = (int)(t < 0 ? t - 0.5 : t + 0.5);
    double r = (x - (double)k * LN2_HI) - (double)k * LN2_LO;
    double term = 1.0, sum = 1.0;
    for (int n = 1; n <= 24; ++n) {
        term = term * r / (double)n;
        sum = sum + term;
    }
    /* split the scaling so pow2i stays in the normal range */
    if (k < -1000) return sum * pow2i(k + 600) * pow2i(-600);
    return sum * pow2i(k);
}

static const double INV_SQRT_2PI = 0.39894228040143267794;

static double det_pdf(double z) { return INV_SQRT_2PI * det_exp(-0.5 * z * z); }

/* Phi(z) for z >= 0: 0.5 + pdf(z) * sum_n z^(2n+1) / (2n+1)!!  */
static double det_cdf_pos(double z) {
    double term = z, sum = z;
    double z2 = z * z;
    for (int n = 1; n < 400; ++n) {
        term = term * z2 / (double)(2 * n + 1);
        sum = sum + term;
        if (term < sum * 1e-18) break;
    }
    return 0.5 + det_pdf(z) * sum;
}

static double g_quant[NQ];
static int g_quant_ready = 0;

static void build_quantiles(void) {
    /* upper half: cells k = NQ/2 .. NQ-1, p_k = (k + 0.5) / NQ, z >= 0 */
    double z = 0.0;
    for (int k = NQ / 2; k < NQ; ++k) {
        double p = ((double)k + 0.5) / (double)NQ;
        for (int it = 0; it < 12; ++it) {
            double f = det_cdf_pos(z) - p;
            z = z - f / det_pdf(z);
            if (z < 0) z = 0;
        }
        g_quant[k] = z;
        g_quant[NQ - 1 - k] = -z;
    }
    g_quant_ready = 1;
}

__attribute__((constructor)) static void grgen_init(void) { build_quantiles(); }

double grgen_quantile(int k) {
    if (k < 0 || k >= NQ) return 0.0;
    return g_quant[k];
}

/* float -> bf16 bits, round to nearest even (NaN kept quiet). */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* out[i] = mean + sigma * Z[word(seed, stream, offset + i) >> 48]
   dtype 0: float32, dtype 1: bf16 bits (uint16). */
void grgen_normal(uint64_t seed, uint64_t stream, double mean, double sigma, int dtype,
                  void *out, int64_t n, int64_t offset) {
    uint64_t key = stream_key(seed, stream);
    if (dtype == 1) {
        uint16_t *o = (uint16_t *)out;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            uint64_t w = mix64(key + (uint64_t)(offset + i + 1) * GAMMA);
            double v = mean + sigma * g_quant[w >> 48];
            o[i] = f32_to_bf16((float)v);
        }
    } else {
        float *o = (float *)out;
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i) {
            uint64_t w = mix64(key + (uint64_t)(offset + i + 1) * GAMMA);
            o[i] = (float)(mean + sigma * g_quant[w >> 48]);
        }
    }
}

/* out[i] uniform in [lo, hi) */
void grgen_ints(uint64_t seed, uint64_t stream, int32_t lo, int32_t hi, int32_t *out, int64_t n,
                int64_t offset) {
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo);
    for (int64_t i = 0; i < n; ++i) {
        uint64_t w = mix64(key + (uint64_t)(offset + i + 1) * GAMMA);
        out[i] = (int32_t)((int64_t)lo + (int64_t)(((w >> 32) * span) >> 32));
    }
}

/* out = a permutation of 0..n-1 (Fisher-Yates driven by word(i)) */
void grgen_permutation(uint64_t seed, uint64_t stream, int32_t *out, int64_t n) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i > 0; --i) {
        uint64_t w = mix64(key + (uint64_t)(i + 1) * GAMMA);
        int64_t j = (int64_t)(((w >> 32) * (uint64_t)(i + 1)) >> 32);
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}
