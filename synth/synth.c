/*
 * Seeded synthetic input generator shared by the CPU oracle and the CUDA path.
 *
 * It holds none of the MLP's arithmetic: it only draws the input tensors
 * (activations, weights, biases, upstream gradients) that both sides consume.
 *
 * Generator: element i of a tensor with seed s takes two 64-bit draws
 *   z_j = mix64(s + (2i + j + 1) * 0x9E3779B97F4A7C15),  j = 0, 1
 * where mix64 is the SplitMix64 output function (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).  The two
 * draws become u1 in (0,1] and u2 in [0,1) with 53-bit resolution and the
 * Box-Muller transform (Box & Muller, 1958) gives one standard normal
 *   n = sqrt(-2 ln u1) * cos(2 pi u2),
 * scaled as mean + std * n and rounded to fp32.  Because every element is a
 * pure function of (seed, index) the generator is counter-based: any slice
 * can be drawn on its own and threads need no shared state.
 *
 * bf16 conversion is round-to-nearest-even on the fp32 bit pattern.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

void synth_normal_f32(uint64_t seed, int64_t offset, int64_t n, double mean,
                      double stddev, float *out) {
    const double two_pi = 6.283185307179586476925286766559;
    const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t idx = (uint64_t)(offset + i);
        uint64_t z1 = mix64(seed + (2 * idx + 1) * GOLDEN_GAMMA);
        uint64_t z2 = mix64(seed + (2 * idx + 2) * GOLDEN_GAMMA);
        double u1 = (double)((z1 >> 11) + 1) * inv53; /* (0, 1] */
        double u2 = (double)(z2 >> 11) * inv53;       /* [0, 1) */
        double g = sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
        out[i] = (float)(mean + stddev * g);
    }
}

void synth_f32_to_bf16(const float *in, uint16_t *out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        union { float f; uint32_t u; } v;
        v.f = in[i];
        uint32_t u = v.u;
        if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) {
            out[i] = (uint16_t)((u >> 16) | 0x0040u); /* quiet NaN */
        } else {
            uint32_t lsb = (u >> 16) & 1u;
            out[i] = (uint16_t)((u + 0x7FFFu + lsb) >> 16);
        }
    }
}

void synth_bf16_to_f32(const uint16_t *in, float *out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        union { float f; uint32_t u; } v;
        v.u = ((uint32_t)in[i]) << 16;
        out[i] = v.f;
    }
}

int synth_num_threads(void) {
    int t = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        t = omp_get_num_threads();
    }
#endif
    return t;
}
