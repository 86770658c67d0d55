/*
 * Seeded synthetic inputs for the tensor-parallel MLP block.
 *
 * This file holds none of the block's arithmetic: it only draws the numbers
 * that both the CPU oracle and the CUDA library consume (X, W1, b1, W2, b2).
 *
 * Generator (counter based, so any element can be drawn independently and in
 * parallel):
 *   mix64(z)      the SplitMix64 output function (Steele, Lea, Flood,
 *                 "Fast splittable pseudorandom number generators", OOPSLA 2014):
 *                 z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27;
 *                 z *= 0x94D049BB133111EB; z ^= z>>31.
 *   key           = mix64(seed * 0x9E3779B97F4A7C15 + stream + 1)
 *   word(c)       = mix64(key + (c + 1) * 0x9E3779B97F4A7C15)   (c = counter)
 *   uniform(c)    = (word(c) >> 11) * 2^-53                      in [0, 1)
 *   normal(e)     = Box-Muller on u1 = 1 - uniform(2e) in (0,1],
 *                   u2 = uniform(2e+1):  sqrt(-2 ln u1) * cos(2 pi u2)
 *   value(e)      = mean + std * normal(e), rounded once from double to
 *                   bfloat16 with round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z) {
    z ^= z >> 30;
    z *= 0xBF58476D1CE4E5B9ull;
    z ^= z >> 27;
    z *= 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z;
}

static inline double uniform01(uint64_t key, uint64_t c) {
    return (double)(mix64(key + (c + 1) * GOLDEN) >> 11) * 0x1.0p-53;
}

/* Round a double to the nearest bfloat16 (ties to even) in one step.
 * Finite values only; the generator never produces inf or nan. */
static inline uint16_t round_to_bf16(double d) {
    uint64_t b;
    memcpy(&b, &d, sizeof b);
    uint64_t sign = b >> 63;
    uint64_t mag = b & 0x7FFFFFFFFFFFFFFFull;
    if (mag == 0) return (uint16_t)(sign << 15);
    int e = (int)(mag >> 52) - 1023; /* unbiased exponent of d */
    if (e >= -126) {
        /* normal bf16 range: keep 7 fraction bits, round the other 45 */
        uint64_t lsb = (mag >> 45) & 1;
        mag += (1ull << 44) - 1 + lsb;
        mag &= ~((1ull << 45) - 1);
        int e2 = (int)(mag >> 52) - 1023;
        if (e2 > 127) return (uint16_t)((sign << 15) | 0x7F80); /* overflow to inf */
        uint32_t bf = (uint32_t)((e2 + 127) << 7) | (uint32_t)((mag >> 45) & 0x7F);
        return (uint16_t)((sign << 15) | bf);
    }
    /* subnormal bf16 range: quantum is 2^-133 */
    double q = ldexp(fabs(d), 133); /* exact scaling */
    double r = nearbyint(q);        /* default rounding mode: ties to even */
    uint32_t m = (uint32_t)r;       /* m <= 128; m == 128 is the smallest normal */
    return (uint16_t)((sign << 15) | m);
}

uint64_t synth_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * GOLDEN + stream + 1);
}

/* n values ~ N(mean, std^2), rounded to bf16, element e drawn from counters 2e, 2e+1
 * (offset by `first`, so a slice of a large tensor can be drawn on its own). */
void synth_normal_bf16(uint64_t seed, uint64_t stream, double mean, double std, int64_t first,
                       int64_t n, uint16_t *out) {
    const uint64_t key = synth_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t e = (uint64_t)(first + i);
        double u1 = 1.0 - uniform01(key, 2 * e);
        double u2 = uniform01(key, 2 * e + 1);
        double z = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[i] = round_to_bf16(mean + std * z);
    }
}

/* Same draw, returned as double (used by the generator's own tests). */
void synth_normal_f64(uint64_t seed, uint64_t stream, double mean, double std, int64_t first,
                      int64_t n, double *out) {
    const uint64_t key = synth_key(seed, stream);
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t e = (uint64_t)(first + i);
        double u1 = 1.0 - uniform01(key, 2 * e);
        double u2 = uniform01(key, 2 * e + 1);
        out[i] = mean + std * (sqrt(-2.0 * log(u1)) * cos(two_pi * u2));
    }
}

/* Exposed for tests of the rounding step. */
void synth_round_bf16(const double *in, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = round_to_bf16(in[i]);
}

uint64_t synth_mix64(uint64_t z) { return mix64(z); }

int synth_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
