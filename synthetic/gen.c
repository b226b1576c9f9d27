/*
 * Seeded synthetic inputs for the batch-invariant exact GEMM.
 *
 * This file holds no arithmetic of the method itself (no accumulation, no
 * scaling, no rounding to bf16/fp32 outputs): it only draws the operand values
 * that the CPU oracle and the CUDA path both consume. Both sides receive the
 * same arrays; neither recomputes them.
 *
 * Generator: counter-based splitmix64. Element i of stream s under seed S is
 *     key  = mix64(S * G + mix64(s + 1))
 *     u(i) = mix64(key + (i + 1) * G)                 G = 0x9E3779B97F4A7C15
 * so every element can be drawn independently (OpenMP-parallel, any order).
 *
 *   uniform integer in [lo, hi]:   lo + ((u >> 32) * (hi - lo + 1)) >> 32
 *   standard normal (Box-Muller):  u1 = ((u(2i) >> 11) + 1) * 2^-53  in (0, 1]
 *                                  u2 =  (u(2i+1) >> 11)     * 2^-53  in [0, 1)
 *                                  z  = sqrt(-2 ln u1) * cos(2 pi u2)
 *   rounded normal int8:           clamp(nearbyint(sigma * z), -clip, clip)
 *   scaled normal fp32:            (float)z * 2^U,  U uniform integer
 *
 * Box-Muller uses the C library's log/cos, so a draw may differ between two
 * libm builds in the last bit of z; every test draws its inputs on the
 * machine where it runs, so nothing depends on that.
 */
#include <math.h>
#include <stdint.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(seed * GAMMA + mix64(stream + 1));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GAMMA); }

static inline int64_t uniform_int(uint64_t u, int64_t lo, int64_t hi) {
    uint64_t range = (uint64_t)(hi - lo + 1);
    return lo + (int64_t)(((u >> 32) * range) >> 32);
}

static inline double std_normal(uint64_t key, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = ((double)((draw(key, 2 * i) >> 11) + 1)) * 0x1p-53;
    double u2 = ((double)(draw(key, 2 * i + 1) >> 11)) * 0x1p-53;
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

void gen_uniform_i8(uint64_t seed, uint64_t stream, int64_t n, int lo, int hi, int8_t* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (int8_t)uniform_int(draw(key, (uint64_t)i), lo, hi);
}

void gen_uniform_i32(uint64_t seed, uint64_t stream, int64_t n, int lo, int hi, int32_t* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)uniform_int(draw(key, (uint64_t)i), lo, hi);
}

void gen_normal_i8(uint64_t seed, uint64_t stream, int64_t n, double sigma, int clip, int8_t* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double v = nearbyint(sigma * std_normal(key, (uint64_t)i));
        if (v > clip) v = clip;
        if (v < -clip) v = -clip;
        out[i] = (int8_t)v;
    }
}

/* N(0, 1) * 2^U with U uniform in [ulo, uhi] (the exponent draws use stream + 1000). */
void gen_normal_pow2_f32(uint64_t seed, uint64_t stream, int64_t n, int ulo, int uhi, float* out) {
    uint64_t key = stream_key(seed, stream);
    uint64_t ukey = stream_key(seed, stream + 1000);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        int u = (int)uniform_int(draw(ukey, (uint64_t)i), ulo, uhi);
        out[i] = ldexpf((float)std_normal(key, (uint64_t)i), u);
    }
}

/* N(0, 1) * 2^U as fp64 (U uniform in [ulo, uhi], exponent draws on stream + 1000). */
void gen_normal_pow2_f64(uint64_t seed, uint64_t stream, int64_t n, int ulo, int uhi, double* out) {
    uint64_t key = stream_key(seed, stream);
    uint64_t ukey = stream_key(seed, stream + 1000);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        int u = (int)uniform_int(draw(ukey, (uint64_t)i), ulo, uhi);
        out[i] = ldexp(std_normal(key, (uint64_t)i), u);
    }
}

/* sigma * N(0, 1) as fp32 (activation-like inputs for the quantizer). */
void gen_normal_f32(uint64_t seed, uint64_t stream, int64_t n, double sigma, float* out) {
    uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(sigma * std_normal(key, (uint64_t)i));
}
