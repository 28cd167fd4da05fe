/*
 * synth.c - seeded, counter-based synthetic inputs.
 *
 * This module draws random numbers and nothing else.  It holds none of the
 * decoder's arithmetic (no quantisation, packing, normalisation or attention):
 * the engine and the CPU oracle both receive its outputs as plain inputs.
 *
 * Generator: SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014; constants as published by Vigna).  The
 * published sequential form is
 *     state += 0x9E3779B97F4A7C15;  return mix(state);
 * so the i-th output (0-based) of a stream that starts at state s is
 * mix(s + (i + 1) * 0x9E3779B97F4A7C15).  Every value below is a pure
 * function of (seed, tensor_id, index); the order in which threads compute
 * them does not matter.
 *
 * Stream start for a tensor:  s(seed, tid) = mix(mix(seed) ^ (tid * 0xD1B54A32D192ED03)).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_start(uint64_t seed, uint64_t tid) {
    return sm64_mix(sm64_mix(seed) ^ (tid * 0xD1B54A32D192ED03ULL));
}

static inline uint64_t draw(uint64_t s, uint64_t i) {
    return sm64_mix(s + (i + 1) * SM64_GAMMA);
}

/* Draws from an explicit starting state (pins the generator to its published form). */
void synth_raw_state(uint64_t state, int64_t n, uint64_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = draw(state, (uint64_t)i);
}

/* Raw 64-bit draws of the stream of (seed, tid). */
void synth_raw_u64(uint64_t seed, uint64_t tid, int64_t n, uint64_t *out) {
    uint64_t s = stream_start(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = draw(s, (uint64_t)i);
}

/* Integer uniform on [lo, hi] by the multiply-shift map of the high 32 bits
 * (Lemire 2019); the bias is below (hi-lo+1)/2^32. */
static inline int64_t map_int(uint64_t x, int64_t lo, int64_t hi) {
    uint64_t range = (uint64_t)(hi - lo + 1);
    return lo + (int64_t)(((x >> 32) * range) >> 32);
}

void synth_randint_i8(uint64_t seed, uint64_t tid, int64_t n, int32_t lo, int32_t hi,
                      int8_t *out) {
    uint64_t s = stream_start(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (int8_t)map_int(draw(s, (uint64_t)i), lo, hi);
}

void synth_randint_i32(uint64_t seed, uint64_t tid, int64_t n, int32_t lo, int32_t hi,
                       int32_t *out) {
    uint64_t s = stream_start(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)map_int(draw(s, (uint64_t)i), lo, hi);
}

/* Uniform float on [a, b) from the top 24 bits. */
void synth_uniform_f32(uint64_t seed, uint64_t tid, int64_t n, float a, float b, float *out) {
    uint64_t s = stream_start(seed, tid);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        double u = (double)(draw(s, (uint64_t)i) >> 40) * (1.0 / 16777216.0);
        out[i] = (float)((double)a + ((double)b - (double)a) * u);
    }
}

/* Normal(mean, std) by the Box-Muller transform (Box & Muller 1958): draws
 * 2j and 2j+1 give u1 in (0,1] and u2 in [0,1); element 2j takes the cosine
 * branch and element 2j+1 the sine branch. */
void synth_normal_f32(uint64_t seed, uint64_t tid, int64_t n, float mean, float std, float *out) {
    uint64_t s = stream_start(seed, tid);
    const double two_pi = 6.283185307179586476925286766559;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint64_t j = (uint64_t)i >> 1;
        double u1 = (double)((draw(s, 2 * j) >> 11) + 1) * (1.0 / 9007199254740992.0);
        double u2 = (double)(draw(s, 2 * j + 1) >> 11) * (1.0 / 9007199254740992.0);
        double r = sqrt(-2.0 * log(u1));
        double z = (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
        out[i] = (float)((double)mean + (double)std * z);
    }
}

/* Storage conversion of generated fp32 values to bfloat16 bit patterns,
 * round-to-nearest-even (inputs are finite). */
void synth_f32_to_bf16(int64_t n, const float *in, uint16_t *out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t b;
        memcpy(&b, &in[i], 4);
        uint32_t r = b + 0x7FFFu + ((b >> 16) & 1u);
        out[i] = (uint16_t)(r >> 16);
    }
}

/* Seeded permutation of 0..n-1 (Fisher-Yates / Durstenfeld), draw i picks
 * the swap partner for position n-1-i. */
void synth_permutation(uint64_t seed, uint64_t tid, int64_t n, int32_t *out) {
    uint64_t s = stream_start(seed, tid);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = 0; i + 1 < n; ++i) {
        int64_t top = n - 1 - i;
        int64_t j = map_int(draw(s, (uint64_t)i), 0, top);
        int32_t t = out[top];
        out[top] = out[j];
        out[j] = t;
    }
}
