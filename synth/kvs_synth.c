/*
 * Seeded synthetic inputs shared by the test harness, the benchmark and the
 * oracle's callers.  This file holds random-number generation only: nothing
 * of the attention method (no quantisation, no softmax) lives here.
 *
 * Generator: SplitMix64 (G. Steele, D. Lea, C. Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014; finaliser constants as
 * published with Java's SplittableRandom).  It is used counter-style: the
 * c-th 64-bit output of stream (seed, tag) is mix(base + (c + 1) * GAMMA)
 * with base = mix(seed ^ mix(tag)), which is exactly the c-th output of a
 * SplitMix64 generator whose state starts at base.  Any element can be
 * produced independently, so fills are split across threads freely and the
 * result does not depend on the thread count.
 *
 * Normal variates: Box-Muller (G. Box, M. Muller, 1958) in fp64 on two
 * uniforms u1 = U(2k), u2 = U(2k+1) in the open interval (0,1); element 2k
 * takes r*cos(2*pi*u2), element 2k+1 takes r*sin(2*pi*u2), r = sqrt(-2 ln u1).
 * The fp64 value is rounded to fp32 (round-to-nearest-even).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t synth_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline uint64_t synth_base(uint64_t seed, uint64_t tag) {
    return synth_mix(seed ^ synth_mix(tag + SYNTH_GAMMA));
}

static inline uint64_t synth_at(uint64_t base, uint64_t c) {
    return synth_mix(base + (c + 1ull) * SYNTH_GAMMA);
}

/* uniform in the open interval (0,1): 53 random bits, offset by half a step */
static inline double synth_u01(uint64_t x) {
    return ((double)(x >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* Raw 64-bit outputs c = offset .. offset+n-1 of stream (seed, tag). */
void synth_u64(uint64_t seed, uint64_t tag, uint64_t offset, uint64_t n, uint64_t *out) {
    const uint64_t base = synth_base(seed, tag);
    #pragma omp parallel for schedule(static) if (n > (1u << 16))
    for (int64_t i = 0; i < (int64_t)n; ++i) out[i] = synth_at(base, offset + (uint64_t)i);
}

/* N(0,1) variates, elements offset .. offset+n-1 of stream (seed, tag), as fp32. */
void synth_normal_f32(uint64_t seed, uint64_t tag, uint64_t offset, uint64_t n, float *out) {
    const uint64_t base = synth_base(seed, tag);
    const double two_pi = 6.283185307179586476925286766559;
    #pragma omp parallel for schedule(static) if (n > (1u << 15))
    for (int64_t i = 0; i < (int64_t)n; ++i) {
        const uint64_t e = offset + (uint64_t)i;
        const uint64_t k = e >> 1;
        const double u1 = synth_u01(synth_at(base, 2 * k));
        const double u2 = synth_u01(synth_at(base, 2 * k + 1));
        const double r = sqrt(-2.0 * log(u1));
        const double z = (e & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
        out[i] = (float)z;
    }
}

/* Uniform fp32 values in [lo, hi): lo + (hi - lo) * U, computed in fp64. */
void synth_uniform_f32(uint64_t seed, uint64_t tag, uint64_t offset, uint64_t n,
                       double lo, double hi, float *out) {
    const uint64_t base = synth_base(seed, tag);
    #pragma omp parallel for schedule(static) if (n > (1u << 16))
    for (int64_t i = 0; i < (int64_t)n; ++i)
        out[i] = (float)(lo + (hi - lo) * synth_u01(synth_at(base, offset + (uint64_t)i)));
}
