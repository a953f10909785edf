/*
 * synth.c - seeded synthetic inputs for the bs=1 decode workloads.
 *
 * This module only draws inputs: weights, norm gains, pre-filled K/V and token
 * ids.  It holds none of the decode arithmetic, and both the CPU oracle and the
 * GPU path receive the arrays it writes.
 *
 * Generator (counter based, so any element can be drawn independently and the
 * fill is trivially parallel):
 *   key      = splitmix64(seed ^ splitmix64(stream))
 *   word(k)  = splitmix64(key + k * 0x9E3779B97F4A7C15)
 * splitmix64 is the finaliser published by Steele, Lea and Flood ("Fast
 * splittable pseudorandom number generators", OOPSLA 2014).
 *
 * Normal values use the Box-Muller transform on the pair k = i / 2:
 *   u1 = ((word(2k) >> 40) + 1) * 2^-24   in (0, 1]
 *   u2 =  (word(2k+1) >> 40)    * 2^-24   in [0, 1)
 *   z  = sqrt(-2 ln u1) * (i even ? cos(2 pi u2) : sin(2 pi u2))   (float)
 *   value = mean + std * z, rounded double -> float -> bf16 (ties to even).
 * Uniform integers use lo + (word(i) % (hi - lo)).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t splitmix64(uint64_t x) {
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return splitmix64(seed ^ splitmix64(stream));
}

static uint64_t word_at(uint64_t key, uint64_t k) {
    return splitmix64(key + k * 0x9E3779B97F4A7C15ull);
}

static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Box-Muller pair k: writes z(2k) and z(2k+1), in float (the values are
 * rounded to bf16 afterwards, so float transcendentals are ample). */
static void normal_pair(uint64_t key, uint64_t k, double* z0, double* z1) {
    const float two_pi = 6.28318530717958647692f;
    float u1 = (float)((word_at(key, 2 * k) >> 40) + 1) * (1.0f / 16777216.0f);
    float u2 = (float)(word_at(key, 2 * k + 1) >> 40) * (1.0f / 16777216.0f);
    float r = sqrtf(-2.0f * logf(u1));
    *z0 = (double)(r * cosf(two_pi * u2));
    *z1 = (double)(r * sinf(two_pi * u2));
}

/* out[i] = bf16(mean + std * N(0,1)_i) for i in [0, n). */
void synth_fill_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, uint64_t stream, double mean, double std) {
    uint64_t key = stream_key(seed, stream);
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < npair; ++k) {
        double z0, z1;
        normal_pair(key, (uint64_t)k, &z0, &z1);
        out[2 * k] = float_to_bf16_rne((float)(mean + std * z0));
        if (2 * k + 1 < n) out[2 * k + 1] = float_to_bf16_rne((float)(mean + std * z1));
    }
}

/* out[i] = float(mean + std * N(0,1)_i); the same draws as the bf16 fill before its bf16 rounding. */
void synth_fill_normal_f32(float* out, int64_t n, uint64_t seed, uint64_t stream, double mean, double std) {
    uint64_t key = stream_key(seed, stream);
    int64_t npair = (n + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < npair; ++k) {
        double z0, z1;
        normal_pair(key, (uint64_t)k, &z0, &z1);
        out[2 * k] = (float)(mean + std * z0);
        if (2 * k + 1 < n) out[2 * k + 1] = (float)(mean + std * z1);
    }
}

/* out[i] = lo + word(i) mod (hi - lo), hi > lo. */
void synth_fill_uniform_i32(int32_t* out, int64_t n, uint64_t seed, uint64_t stream, int32_t lo, int32_t hi) {
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)((int64_t)lo + (int64_t)(word_at(key, (uint64_t)i) % span));
}
