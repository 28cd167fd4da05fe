// pack.cpp - offline weight packer (host memory, no GPU).
//
// INT4 ValueShuffle ("How To Construct Your Personal LLM Runtime From Scratch",
// §7): the eight codes of an octet go to bit shifts 0,16,4,20,8,24,12,28, so
// even lanes fill the low half-word and odd lanes the high half-word.  The
// decode kernels then turn each half-word pair (c_2j, c_2j+1) into an exact
// fp16 pair with one lop3 and one fp16 add/fma.
//
// Quantizers (same file: they feed the packer):
//   INT4 group 128 ("How To Construct Your Personal LLM Runtime From Scratch",
//   §3): symmetric, zero point 0, one scale per (output row, group of 128
//   along K), scale = absmax / 7, kept as bfloat16.
//   INT8 per row ("FlashQwen", Stage 8): symmetric, one fp32 scale per output
//   row, computed at load.
// Each code is the fp32 quotient weight / scale rounded half to even, with the
// scale as stored (so that code * scale is the dequantized weight), clamped
// to the format's range; a group or row of zeros gets scale 0 and codes 0.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/llm.h"

namespace {

// bfloat16 of a finite float, rounded to nearest, ties to even (the 16 dropped bits).
uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
float bf16_to_f32(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return f;
}
int clampi(float v, int lo, int hi) { return v < (float)lo ? lo : (v > (float)hi ? hi : (int)v); }

}  // namespace

extern "C" {

int llm_pack_int4_g128(const int8_t *codes, int64_t N, int64_t K, uint32_t *words) {
    if (!codes || !words || N <= 0 || K <= 0 || K % 128 != 0) return LLM_ERR_ARG;
    static const int kShift[8] = {0, 16, 4, 20, 8, 24, 12, 28};
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n) {
        const int8_t *row = codes + n * K;
        uint32_t *out = words + n * (K / 8);
        for (int64_t w = 0; w < K / 8; ++w) {
            uint32_t word = 0;
            for (int i = 0; i < 8; ++i) {
                const int c = row[w * 8 + i];
                bad |= (c < -8 || c > 7);
                word |= ((uint32_t)c & 0xFu) << kShift[i];
            }
            out[w] = word;
        }
    }
    return bad ? LLM_ERR_ARG : LLM_OK;
}

int llm_pack_int8_row(const int8_t *codes, int64_t N, int64_t K, int8_t *out) {
    if (!codes || !out || N <= 0 || K <= 0) return LLM_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t i = 0; i < N * K; ++i) {
        bad |= codes[i] == -128;
        out[i] = codes[i];
    }
    return bad ? LLM_ERR_ARG : LLM_OK;
}

int llm_quantize_int4_g128(const float *w, int64_t N, int64_t K, int8_t *codes, uint16_t *scales) {
    if (!w || !codes || !scales || N <= 0 || K <= 0 || K % 128 != 0) return LLM_ERR_ARG;
    const int64_t G = K / 128;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t g = 0; g < G; ++g) {
            const float *x = w + n * K + g * 128;
            int8_t *c = codes + n * K + g * 128;
            float amax = 0.f;
            for (int i = 0; i < 128; ++i) {
                bad |= !std::isfinite(x[i]);
                amax = std::fmax(amax, std::fabs(x[i]));
            }
            const uint16_t sb = f32_to_bf16_rne(amax / 7.0f);
            scales[n * G + g] = sb;
            const float sc = bf16_to_f32(sb);
            for (int i = 0; i < 128; ++i) c[i] = sc > 0.f ? (int8_t)clampi(std::nearbyint(x[i] / sc), -8, 7) : 0;
        }
    }
    return bad ? LLM_ERR_ARG : LLM_OK;
}

int llm_quantize_int8_row(const float *w, int64_t N, int64_t K, int8_t *codes, float *scales) {
    if (!w || !codes || !scales || N <= 0 || K <= 0) return LLM_ERR_ARG;
    int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (int64_t n = 0; n < N; ++n) {
        const float *x = w + n * K;
        int8_t *c = codes + n * K;
        float amax = 0.f;
        for (int64_t k = 0; k < K; ++k) {
            bad |= !std::isfinite(x[k]);
            amax = std::fmax(amax, std::fabs(x[k]));
        }
        const float sc = amax / 127.0f;
        scales[n] = sc;
        for (int64_t k = 0; k < K; ++k) c[k] = sc > 0.f ? (int8_t)clampi(std::nearbyint(x[k] / sc), -127, 127) : 0;
    }
    return bad ? LLM_ERR_ARG : LLM_OK;
}

}  // extern "C"
