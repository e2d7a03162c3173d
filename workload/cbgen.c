/*
 * Seeded, counter-based input generator for synthetic CacheBlend workloads.
 *
 * This file holds no arithmetic of the blend method: it only turns
 * (seed, stream, index) into numbers.  Both the CPU oracle and the GPU path
 * consume the arrays it writes, so neither side generates its own inputs.
 *
 * Definition (so any element can be recomputed independently):
 *   mix(z)        SplitMix64 finaliser (Steele, Lea & Flood, "Fast splittable
 *                 pseudorandom number generators", OOPSLA 2014):
 *                   z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                   z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                   z =  z ^ (z >> 31)
 *   GAMMA         0x9E3779B97F4A7C15 (the SplitMix64 increment)
 *   key(s, t)     mix(mix(s ^ 0x5851F42D4C957F2D) + t * GAMMA)
 *   draw(s,t,i)   mix(key(s,t) + (i + 1) * GAMMA)      i = 0, 1, 2, ...
 *   unif(x)       (x >> 11) * 2^-53                      in [0, 1)
 *   normal pair p from u1 = 1 - unif(draw(2p)), u2 = unif(draw(2p+1)):
 *                 r = sqrt(-2 ln u1);  z[2p] = r cos(2 pi u2);  z[2p+1] = r sin(2 pi u2)
 *                 (Box & Muller, Ann. Math. Stat. 29, 1958)
 *   value[i]      (float)(std * z[i]) rounded to nearest even, then, for
 *                 bf16 outputs, rounded to nearest even to bfloat16.
 *   token[i]      draw(i) mod vocab
 *   permutation   Fisher-Yates: for i = n-1 .. 1: j = draw(i) mod (i+1); swap(a[i], a[j])
 *
 * Build: gcc -O2 -fopenmp -fPIC -shared (portable C99, no ISA intrinsics).
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <string.h>

#define CBGEN_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t cbgen_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t cbgen_key(uint64_t seed, uint64_t stream) {
    return cbgen_mix(cbgen_mix(seed ^ 0x5851F42D4C957F2DULL) + stream * CBGEN_GAMMA);
}

uint64_t cbgen_draw(uint64_t key, uint64_t i) {
    return cbgen_mix(key + (i + 1) * CBGEN_GAMMA);
}

static inline double cbgen_unif(uint64_t x) {
    return (double)(x >> 11) * (1.0 / 9007199254740992.0);
}

static inline uint16_t cbgen_f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

static inline void cbgen_normal_pair(uint64_t key, uint64_t p, double* z0, double* z1) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = 1.0 - cbgen_unif(cbgen_draw(key, 2 * p));
    double u2 = cbgen_unif(cbgen_draw(key, 2 * p + 1));
    double r = sqrt(-2.0 * log(u1)), s, c;
    sincos(two_pi * u2, &s, &c);
    *z0 = r * c;
    *z1 = r * s;
}

/* Elements [first, first + n) of stream (seed, stream), std * N(0,1): one Box-Muller pair per step. */
#define CBGEN_NORMAL_LOOP(STORE)                                                      \
    const uint64_t key = cbgen_key(seed, stream);                                     \
    const int64_t p0 = first >> 1, p1 = (first + n + 1) >> 1;                         \
    _Pragma("omp parallel for schedule(static)")                                      \
    for (int64_t p = p0; p < p1; ++p) {                                               \
        double z[2];                                                                  \
        cbgen_normal_pair(key, (uint64_t)p, &z[0], &z[1]);                            \
        for (int h = 0; h < 2; ++h) {                                                 \
            int64_t e = 2 * p + h - first;                                            \
            if (e >= 0 && e < n) STORE;                                               \
        }                                                                             \
    }

void cbgen_normal_f32(uint64_t seed, uint64_t stream, int64_t first, int64_t n, double std, float* out) {
    CBGEN_NORMAL_LOOP(out[e] = (float)(std * z[h]))
}

/* Same values, rounded once more to bfloat16 (bit patterns). */
void cbgen_normal_bf16(uint64_t seed, uint64_t stream, int64_t first, int64_t n, double std, uint16_t* out) {
    CBGEN_NORMAL_LOOP(out[e] = cbgen_f32_to_bf16_rne((float)(std * z[h])))
}

/* Constant fill (norm gains), bf16 bit patterns. */
void cbgen_fill_bf16(int64_t n, float value, uint16_t* out) {
    uint16_t b = cbgen_f32_to_bf16_rne(value);
    #pragma omp parallel for schedule(static)
    for (int64_t e = 0; e < n; ++e) out[e] = b;
}

/* Uniform token ids in [0, vocab). */
void cbgen_tokens(uint64_t seed, uint64_t stream, int64_t n, int64_t vocab, int32_t* out) {
    const uint64_t key = cbgen_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)(cbgen_draw(key, (uint64_t)i) % (uint64_t)vocab);
}

/* A seeded permutation of 0..n-1 (Fisher-Yates). */
void cbgen_permutation(uint64_t seed, uint64_t stream, int64_t n, int32_t* out) {
    const uint64_t key = cbgen_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i >= 1; --i) {
        int64_t j = (int64_t)(cbgen_draw(key, (uint64_t)i) % (uint64_t)(i + 1));
        int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}
