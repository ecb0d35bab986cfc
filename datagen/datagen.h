/*
 * datagen.h -- seeded, counter-based synthetic input values.
 *
 * This header is the one piece of code shared by the CUDA library's tests and
 * bench and by the CPU oracle's harness: it turns (seed, stream, counter) into
 * input values, and holds none of the gradient-reduction arithmetic.  The same
 * functions compile for the host (gcc) and the device (nvcc), so an input
 * generated on the GPU and the same input generated on the host are bit-equal.
 *
 * Generator: the SplitMix64 output function (G. Steele, D. Lea, C. Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014), used in
 * counter mode: draw(key, i) = mix64(key + i * golden_gamma).
 *
 * Value recipes (all steps exact integer or single IEEE fp32 operations):
 *  - normal(sigma): Irwin-Hall sum of twelve 16-bit uniform fields taken from
 *    three draws, centred by subtracting its mean 12 * 65535 / 2 = 393210, then
 *    one fp32 multiply by scale = sigma * 2^-16.  Tails are cut at about +-6
 *    sigma; mean 0, standard deviation sigma * sqrt((65536^2 - 1) / 65536^2).
 *  - uniform[-1, 1): the top 24 bits of one draw, minus 2^23, times 2^-23.
 *  - bf16 values are made by truncating the fp32 value's low 16 bits (round
 *    toward zero), which keeps them away from the round-to-nearest-even cast
 *    that the reduction itself performs.
 */
#ifndef DATAGEN_H
#define DATAGEN_H

#include <stdint.h>

#if defined(__CUDACC__)
#define DG_FN static inline __host__ __device__
#else
#define DG_FN static inline
#endif

#define DG_GAMMA 0x9E3779B97F4A7C15ull

DG_FN uint64_t dg_mix64(uint64_t z) {
    z += DG_GAMMA;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* Key of one stream of values, e.g. one replica row of one micro-batch. */
DG_FN uint64_t dg_key(uint64_t seed, uint64_t stream) {
    return dg_mix64(dg_mix64(seed) ^ (stream * 0xD1B54A32D192ED03ull));
}

DG_FN uint64_t dg_draw(uint64_t key, uint64_t counter) {
    return dg_mix64(key + counter * DG_GAMMA);
}

DG_FN uint32_t dg_f32_bits(float f) {
    union { float f; uint32_t u; } c;
    c.f = f;
    return c.u;
}

DG_FN float dg_bits_f32(uint32_t u) {
    union { float f; uint32_t u; } c;
    c.u = u;
    return c.f;
}

/* Sum of the four 16-bit fields of a 64-bit draw. */
DG_FN int32_t dg_sum16x4(uint64_t d) {
    return (int32_t)(d & 0xFFFF) + (int32_t)((d >> 16) & 0xFFFF) +
           (int32_t)((d >> 32) & 0xFFFF) + (int32_t)(d >> 48);
}

/* Irwin-Hall integer in [-393210, 393210] for element i of a stream. */
DG_FN int32_t dg_irwin_hall(uint64_t key, uint64_t i) {
    int32_t s = dg_sum16x4(dg_draw(key, 3 * i)) + dg_sum16x4(dg_draw(key, 3 * i + 1)) +
                dg_sum16x4(dg_draw(key, 3 * i + 2));
    return s - 393210;
}

/* Approximately normal fp32 value; scale must be sigma * 2^-16 (see dg_normal_scale). */
DG_FN float dg_normal_f32(uint64_t key, uint64_t i, float scale) {
#if defined(__CUDA_ARCH__)
    return __fmul_rn((float)dg_irwin_hall(key, i), scale);
#else
    return (float)dg_irwin_hall(key, i) * scale;
#endif
}

DG_FN uint16_t dg_normal_bf16(uint64_t key, uint64_t i, float scale) {
    return (uint16_t)(dg_f32_bits(dg_normal_f32(key, i, scale)) >> 16);
}

/* Uniform fp32 value in [-1, 1), a multiple of 2^-23. */
DG_FN float dg_uniform_f32(uint64_t key, uint64_t i) {
    int32_t u = (int32_t)(dg_draw(key, i) >> 40) - 8388608;
#if defined(__CUDA_ARCH__)
    return __fmul_rn((float)u, 1.0f / 8388608.0f);
#else
    return (float)u * (1.0f / 8388608.0f);
#endif
}

DG_FN uint16_t dg_uniform_bf16(uint64_t key, uint64_t i) {
    return (uint16_t)(dg_f32_bits(dg_uniform_f32(key, i)) >> 16);
}

/* Integer in [lo, lo + span) from one draw (used for parameter sizes). */
DG_FN int64_t dg_int_range(uint64_t key, uint64_t i, int64_t lo, int64_t span) {
    return lo + (int64_t)(dg_draw(key, i) % (uint64_t)span);
}

/* Value kinds understood by the fill functions. */
enum { DG_NORMAL = 0, DG_UNIFORM = 1 };
/* Element types understood by the fill functions. */
enum { DG_BF16 = 0, DG_F32 = 1 };

#endif /* DATAGEN_H */
