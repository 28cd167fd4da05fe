/* Plain C99 use of the C ABI (host-only calls): the headers compile as C, the
 * symbols link with C linkage, and the quantizer, packer and model-file size
 * behave as documented.  Prints "ok" and exits 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "llm.h"
#include "llm_ops.h"

#define CHECK(c)                                              \
    do {                                                      \
        if (!(c)) {                                           \
            fprintf(stderr, "failed: %s (line %d)\n", #c, __LINE__); \
            return 1;                                         \
        }                                                     \
    } while (0)

int main(void) {
    float w[2 * 128];
    int8_t codes[2 * 128];
    uint16_t scales[2];
    uint32_t words[2 * 16];
    int i;
    for (i = 0; i < 256; ++i) w[i] = (float)((i % 15) - 7) * 0.5f; /* absmax 3.5: scale 0.5 */
    CHECK(llm_quantize_int4_g128(w, 2, 128, codes, scales) == LLM_OK);
    CHECK(scales[0] == 0x3F00 && scales[1] == 0x3F00);             /* bf16 0.5 */
    for (i = 0; i < 256; ++i) CHECK(codes[i] == (i % 15) - 7);
    CHECK(llm_pack_int4_g128(codes, 2, 128, words) == LLM_OK);
    CHECK(llm_quantize_int4_g128(w, 2, 100, codes, scales) == LLM_ERR_ARG);

    llm_config c;
    memset(&c, 0, sizeof c);
    c.n_layers = 2; c.hidden = 256; c.n_q_heads = 4; c.n_kv_heads = 2; c.head_dim = 64;
    c.mlp = 768; c.vocab = 1024; c.rms_eps = 1e-6f; c.rope_base = 1e6f; c.qkv_bias = 1;
    c.weight_format = LLM_FMT_INT4_G128; c.layout_id = LLM_LAYOUT_INT4_VALUESHUFFLE;
    c.max_context = 256; c.page_tokens = 16;
    int64_t bytes = 0;
    CHECK(llm_model_file_bytes(&c, &bytes) == LLM_OK && bytes > 256 && bytes % 2 == 0);
    llm_config r;
    CHECK(llm_model_file_read_config("/nonexistent/file.qd", &r) == LLM_ERR_IO);
    CHECK(strlen(llm_status_str(LLM_ERR_FORMAT)) > 0);
    printf("ok\n");
    return 0;
}
