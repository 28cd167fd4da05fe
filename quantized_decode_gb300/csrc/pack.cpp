// pack.cpp - offline weight packer (host memory, no GPU).
//
// INT4 ValueShuffle ("How To Construct Your Personal LLM Runtime From Scratch",
// §7): the eight codes of an octet go to bit shifts 0,16,4,20,8,24,12,28, so
// even lanes fill the low half-word and odd lanes the high half-word.  The
// decode kernels then turn each half-word pair (c_2j, c_2j+1) into an exact
// fp16 pair with one lop3 and one fp16 add/fma.
#include <cstdint>
#include <cstring>

#include "../../include/llm.h"

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

}  // extern "C"
