/*
 * Seeded synthetic inputs for NA3D: iid N(0,1) values rounded to bf16.
 *
 * This file holds random-number generation only, none of the attention
 * arithmetic. Both the CPU oracle and the CUDA path consume what it writes.
 *
 * Generator (counter based, so any element can be drawn independently and in
 * parallel):
 *   - splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): the k-th output of the stream seeded with
 *     `seed` is mix(seed + (k + 1) * 0x9E3779B97F4A7C15).
 *   - uniform u in (0,1): ((x >> 11) + 0.5) * 2^-53, never 0 or 1.
 *   - Box-Muller (1958) on the pair (u[2j], u[2j+1]):
 *       r = sqrt(-2 ln u[2j]), z[2j] = r cos(2 pi u[2j+1]), z[2j+1] = r sin(2 pi u[2j+1]).
 *   - value i of a request with counter base c0 is z[c0 + i], computed in
 *     fp64, then rounded to fp32, optionally multiplied by an fp32 scale (the
 *     head_dim^-0.5 pre-scale of q), then rounded once to bf16 (nearest even).
 *
 * libm's log/cos/sin may differ in the last ulp between machines; after the
 * bf16 rounding that almost never shows. Every consumer generates its inputs
 * on the machine it runs on, so nothing depends on cross-machine equality.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t sm64_at(uint64_t seed, uint64_t k) {
    uint64_t z = seed + (k + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static inline double uniform_at(uint64_t seed, uint64_t k) {
    return ((double)(sm64_at(seed, k) >> 11) + 0.5) * 0x1.0p-53;
}

static inline double normal_at(uint64_t seed, uint64_t n) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t j = n >> 1;
    double u1 = uniform_at(seed, 2 * j);
    double u2 = uniform_at(seed, 2 * j + 1);
    double r = sqrt(-2.0 * log(u1));
    return (n & 1u) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

/* out[i] = bf16(fp32(z[c0+i]) * scale) for i in [0, n); scale is applied only
 * when apply_scale != 0. nthreads <= 0 uses the OpenMP default. */
void na3d_gen_normal_bf16(uint64_t seed, uint64_t c0, int64_t n, float scale,
                          int apply_scale, uint16_t* out, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) {
#pragma omp parallel for schedule(static) num_threads(nthreads)
        for (int64_t i = 0; i < n; ++i) {
            float f = (float)normal_at(seed, c0 + (uint64_t)i);
            if (apply_scale) f = f * scale;
            out[i] = f32_to_bf16_rne(f);
        }
        return;
    }
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) {
        float f = (float)normal_at(seed, c0 + (uint64_t)i);
        if (apply_scale) f = f * scale;
        out[i] = f32_to_bf16_rne(f);
    }
}

/* fp64 normals, for tests of the generator itself. */
void na3d_gen_normal_f64(uint64_t seed, uint64_t c0, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = normal_at(seed, c0 + (uint64_t)i);
}
