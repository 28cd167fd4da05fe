// ops.cu - single-kernel entry points (llm_ops.h): the engine's own kernels,
// launched one at a time on the caller's stream.  Scratch that a kernel needs
// (attention partials, argmax slots, arrival counters) is stream-ordered
// (cudaMallocAsync / cudaFreeAsync) and zeroed where it must start at zero.
#include <cmath>

#include "../../include/llm.h"
#include "../../include/llm_ops.h"
#include "kernels.h"
#include "ops_util.h"
#include "prefill.h"

using namespace qd;

namespace {

LaunchCfg op_cfg(void *stream) {
    LaunchCfg lc{};
    lc.stream = (cudaStream_t)stream;
    lc.pdl = false;
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&lc.n_sm, cudaDevAttrMultiProcessorCount, dev);
    return lc;
}

bool a16(const void *p) { return p && ((uintptr_t)p & 15) == 0; }

int status(cudaError_t e) { return e == cudaSuccess ? LLM_OK : LLM_ERR_CUDA; }

}  // namespace

extern "C" {

int llm_op_gemv_int4(const void *w, const void *s, const void *bias, int32_t N, int32_t K,
                     const float *x, float *y, void *stream) {
    if (!a16(w) || !s || !a16(x) || !y || N <= 0 || K <= 0 || N % 32 || K % 256) return LLM_ERR_ARG;
    if (!gemv_shape_ok(kFmtInt4, N, K, 0)) return LLM_ERR_ARG;
    GemvArgs a{};
    a.mode = 0; a.w = w; a.s = s; a.bias = (const uint16_t *)bias; a.N = N; a.K = K; a.x = x; a.y = y;
    return status(launch_gemv(op_cfg(stream), kFmtInt4, a));
}

int llm_op_gemv_int4_a8(const void *w, const void *s, int32_t N, int32_t K, const float *x, float *y,
                        void *stream) {
    if (!a16(w) || !s || !a16(x) || !y || N <= 0 || K <= 0 || N % 32 || K % 256) return LLM_ERR_ARG;
    if (!gemv_shape_ok(kFmtInt4A8, N, K, 0)) return LLM_ERR_ARG;
    GemvArgs a{};
    a.mode = 0; a.w = w; a.s = s; a.N = N; a.K = K; a.x = x; a.y = y;
    return status(launch_gemv(op_cfg(stream), kFmtInt4A8, a));
}

int llm_op_gemv_int8(const void *w, const float *s, int32_t N, int32_t K, const float *x, float *y,
                     void *stream) {
    if (!a16(w) || !s || !a16(x) || !y || N <= 0 || K <= 0 || N % 32 || K % 128) return LLM_ERR_ARG;
    if (!gemv_shape_ok(kFmtInt8, N, K, 0)) return LLM_ERR_ARG;
    GemvArgs a{};
    a.mode = 0; a.w = w; a.s = s; a.N = N; a.K = K; a.x = x; a.y = y;
    return status(launch_gemv(op_cfg(stream), kFmtInt8, a));
}

int llm_op_sample(const float *logits, int32_t V, float temperature, int32_t top_k, float top_p,
                  uint64_t seed, uint64_t counter, int32_t *token, void *stream) {
    if (!logits || !token || V < 1 || !(temperature > 0.f) || !(temperature < INFINITY) || top_k < 1 ||
        top_k > kMaxTopK || top_k > V || !(top_p > 0.f) || top_p > 1.f)
        return LLM_ERR_ARG;
    LaunchCfg lc = op_cfg(stream);
    SampleArgs a{};
    a.logits = logits; a.V = V; a.temperature = temperature; a.top_k = top_k; a.top_p = top_p;
    a.seed = seed; a.counter = counter; a.token_out = token; a.st = nullptr; a.advance = 0;
    return status(launch_sample(lc, a));
}

int llm_op_lm_head_argmax(const void *w, const float *lm_scale, const void *gamma, float eps,
                          int32_t N, int32_t K, const float *x, float *logits, int32_t *token,
                          void *stream) {
    const int fmt = lm_scale ? kFmtInt8 : kFmtBf16;
    if (!a16(w) || !a16(gamma) || !a16(x) || !logits || !token || N <= 0 || N % 64 || K % 256)
        return LLM_ERR_ARG;
    if (!lm_head_shape_ok(fmt, N, K)) return LLM_ERR_ARG;
    LaunchCfg lc = op_cfg(stream);
    const int grid = lm_head_grid(lc, N);
    char *scratch = nullptr;
    const size_t bytes = (size_t)grid * 8 + 16;
    if (cudaMallocAsync((void **)&scratch, bytes, lc.stream) != cudaSuccess) return LLM_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, 16, lc.stream) != cudaSuccess) return LLM_ERR_CUDA;
    LmHeadArgs a{};
    a.fmt = fmt; a.w = w; a.scale = lm_scale; a.gamma = (const uint16_t *)gamma; a.eps = eps;
    a.N = N; a.K = K; a.x = x; a.logits = logits;
    a.counter = (int *)scratch;
    a.part_val = (float *)(scratch + 16);
    a.part_idx = (int *)(scratch + 16 + (size_t)grid * 4);
    a.token_out = token; a.st = nullptr; a.advance = 0;
    cudaError_t e = launch_lm_head(lc, a, grid);
    cudaError_t f = cudaFreeAsync(scratch, lc.stream);
    return status(e != cudaSuccess ? e : f);
}

int llm_op_attention(const float *q, const void *k_pool, const void *v_pool, const int32_t *page_table,
                     int32_t n_pool_pages, int32_t T, int32_t Hq, int32_t Hkv, int32_t d, int32_t n_splits,
                     float *out, void *stream) {
    if (!q || !a16(k_pool) || !a16(v_pool) || !page_table || !out || T < 1 || Hkv < 1 ||
        Hq % Hkv || Hq / Hkv > kMaxGqa || (d != 64 && d != 128) || n_splits < 0 || n_splits > 256 ||
        !op_pool_pages_ok(n_pool_pages, Hkv))
        return LLM_ERR_ARG;
    LaunchCfg lc = op_cfg(stream);
    const int n_pg = (T + kPageTokens - 1) / kPageTokens;
    const int cs = attention_split_multiple();
    const int P = n_splits ? (n_splits + cs - 1) / cs * cs : default_splits(lc.n_sm, Hq, Hkv, d, n_pg);
    if (P > 256) return LLM_ERR_ARG;
    const int G = Hq / Hkv;
    const size_t o_bytes = (size_t)Hkv * P * G * d * 4, ml_bytes = (size_t)Hkv * P * G * 2 * 4;
    const size_t cnt_bytes = 256;  // Hkv counters + error word
    if (Hkv + 1 > (int)(cnt_bytes / 4)) return LLM_ERR_ARG;
    char *scratch = nullptr;
    if (cudaMallocAsync((void **)&scratch, cnt_bytes + o_bytes + ml_bytes, lc.stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    if (cudaMemsetAsync(scratch, 0, cnt_bytes, lc.stream) != cudaSuccess) return LLM_ERR_CUDA;
    AttnArgs a{};
    a.q = q; a.k_pool = (const uint16_t *)k_pool; a.v_pool = (const uint16_t *)v_pool;
    a.page_table = page_table; a.n_pages = n_pool_pages;
    a.st = nullptr; a.T_fixed = T;
    a.Hq = Hq; a.Hkv = Hkv; a.d = d; a.P = P;
    a.counter = (int *)scratch;
    a.err = (int *)scratch + Hkv;
    a.part_o = (float *)(scratch + cnt_bytes);
    a.part_ml = (float *)(scratch + cnt_bytes + o_bytes);
    a.out = out;
    cudaError_t e = launch_attention(lc, a);
    int rc = e == cudaSuccess ? op_read_err(a.err, lc.stream) : LLM_ERR_CUDA;
    cudaError_t f = cudaFreeAsync(scratch, lc.stream);
    return rc != LLM_OK ? rc : status(f);
}

int llm_op_dequant_f16(int32_t fmt, const void *w, const void *s, int32_t N, int32_t K, void *out,
                       void *stream) {
    if (!a16(w) || !s || !a16(out) || N <= 0 || K <= 0) return LLM_ERR_ARG;
    if (fmt == LLM_FMT_INT4_G128 ? K % 128 != 0 : (fmt != LLM_FMT_INT8_ROW || K % 8 != 0)) return LLM_ERR_ARG;
    DequantArgs a{};
    a.fmt = fmt == LLM_FMT_INT4_G128 ? kFmtInt4 : kFmtInt8;
    a.w = w; a.s = s; a.N = N; a.K = K; a.out = (uint16_t *)out;
    LaunchCfg lc = op_cfg(stream);
    return status(launch_dequant(lc.stream, lc.n_sm, a));
}

int llm_op_gemm_f16(const void *A, const void *B, int32_t M, int32_t N, int32_t K, float *C, void *stream) {
    if (!a16(A) || !a16(B) || !a16(C) || M <= 0 || N <= 0 || K <= 0 || N % kTcBN || K % kTcBK) return LLM_ERR_ARG;
    CUtensorMap am, bm;
    if (tc_operand_map(&am, A, (uint64_t)M, (uint64_t)K) != cudaSuccess ||
        tc_operand_map(&bm, B, (uint64_t)N, (uint64_t)K) != cudaSuccess)
        return LLM_ERR_CUDA;
    TcGemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.mode = kEpiStore; a.c = C; a.ldc = N; a.wait_ns = 1000000000ull;
    return status(launch_tc_gemm((cudaStream_t)stream, am, bm, a));
}

int llm_op_gemm_quant(int32_t fmt, const void *A, const void *w, const void *s, int32_t M, int32_t N, int32_t K,
                      float *C, void *stream) {
    if (!a16(A) || !a16(w) || !s || !a16(C) || M <= 0 || N <= 0 || K <= 0 || N % kTcBN || K % 128) return LLM_ERR_ARG;
    if (fmt != LLM_FMT_INT4_G128 && fmt != LLM_FMT_INT8_ROW) return LLM_ERR_ARG;
    const int f = fmt == LLM_FMT_INT4_G128 ? kFmtInt4 : kFmtInt8;
    CUtensorMap am, wm[3];
    if (tc_act_map(&am, A, (uint64_t)M, (uint64_t)K) != cudaSuccess ||
        tc_weight_map(&wm[0], w, f, (uint64_t)N, (uint64_t)K, kTcBN) != cudaSuccess)
        return LLM_ERR_CUDA;
    wm[1] = wm[2] = wm[0];
    TcQuantB b{};
    b.fmt = f; b.interleave = 0; b.n_seg = 1; b.seg_rows[0] = N; b.scale[0] = s;
    TcGemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.mode = kEpiStore; a.c = C; a.ldc = N; a.wait_ns = 1000000000ull;
    return status(launch_tc_gemm_q((cudaStream_t)stream, am, wm, b, a));
}

}  // extern "C"
