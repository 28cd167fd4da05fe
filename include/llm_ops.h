/*
 * llm_ops.h - single kernels of the decode step behind the C ABI (libllm.so).
 *
 * These run exactly the device code the engine's captured step runs, one
 * kernel at a time, so each can be checked against the CPU oracle on its own.
 * All array arguments are DEVICE pointers (16-byte aligned where they hold
 * weights); `stream` is a cudaStream_t or NULL for the legacy default stream.
 * Calls are asynchronous on `stream`; launch-time errors are returned as
 * LLM_ERR_CUDA, argument errors as LLM_ERR_ARG (codes from llm.h).
 */
#ifndef QD_LLM_OPS_H
#define QD_LLM_OPS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* y[n] = sum_k code[n][k] * scale[n][k/128] * x[k] (+ bias[n]) for n < N.
 * INT4 group-128 dequant GEMV ("How To Construct Your Personal LLM Runtime From
 * Scratch", §7: mask 4 bits, sign-extend bit 3, multiply by the group scale,
 * accumulate the row in FP32).  w: layout LLM_LAYOUT_INT4_VALUESHUFFLE words
 * [N][K/8]; s: bf16 [N][K/128]; bias: bf16 [N] or NULL; x: fp32 [K]; y: fp32 [N].
 * N % 32 == 0, K % 256 == 0.                                               */
/* The same product on int8 activations ("How To Construct Your Personal LLM
 * Runtime From Scratch", §7, Path A: activations quantized to INT8 with one
 * scale per group before the GEMV, __dp4a products, the group scales applied
 * in the accumulator).  For each group g of 128 along K: sx[g] = max|x| / 127
 * and q[k] = x[k] / sx[g] rounded half to even (fp32, clamped to +-127; a zero
 * group has sx 0 and codes 0), and
 *   y[n] = sum_g scale[n][g] * sx[g] * sum_{k in g} code[n][k] * q[k],
 * the inner sums exact in int32.  Arguments as llm_op_gemv_int4 (no bias).
 * N % 32 == 0, K % 256 == 0, K <= 32768.                                    */
int llm_op_gemv_int4_a8(const void *w, const void *s, int32_t N, int32_t K, const float *x, float *y,
                        void *stream);

int llm_op_gemv_int4(const void *w, const void *s, const void *bias, int32_t N, int32_t K,
                     const float *x, float *y, void *stream);

/* y[n] = scale[n] * sum_k code[n][k] * x[k] ("FlashQwen", stage 8: INT8 codes
 * with one scale per output row).  w: int8 [N][K]; s: fp32 [N].
 * N % 32 == 0, K % 128 == 0.                                               */
int llm_op_gemv_int8(const void *w, const float *s, int32_t N, int32_t K, const float *x,
                     float *y, void *stream);

/* LM head with fused greedy argmax ("FlashQwen", stage 5): n = RMSNorm(x) with
 * gain gamma (bf16 [K]) and eps; logits[v] = W[v] . n for v < N with W bf16
 * [N][K] (lm_scale == NULL) or int8 [N][K] times lm_scale fp32 [N]; *token =
 * the lowest index of the maximum logit.  N % 64 == 0, K % 256 == 0.
 * token: int32 DEVICE pointer.                                             */
int llm_op_lm_head_argmax(const void *w, const float *lm_scale, const void *gamma, float eps,
                          int32_t N, int32_t K, const float *x, float *logits, int32_t *token,
                          void *stream);

/* The decode step's sampler on given logits (see llm_set_sampling in llm.h):
 * logits fp32 [V] and token (one int32) are device pointers; the draw uses
 * counter as its number.  temperature > 0, 1 <= top_k <= min(V, 1024),
 * 0 < top_p <= 1; otherwise LLM_ERR_ARG.                                     */
int llm_op_sample(const float *logits, int32_t V, float temperature, int32_t top_k, float top_p,
                  uint64_t seed, uint64_t counter, int32_t *token, void *stream);

/* Split-K grouped-query decode attention over a paged bf16 KV cache with the
 * log-sum-exp combine ("FlashQwen", stage 7; GQA per "Bare-Metal LLM Inference
 * on NVIDIA H100", "Architectural Blueprint").  For every query head h with
 * group g = h / (Hq/Hkv): out[h] = sum_t softmax_t(q_h . K[g][t] / sqrt(d)) V[g][t]
 * over t < T.  q: fp32 [Hq][d] (already rotated); k_pool, v_pool: bf16
 * [n_pool_pages][Hkv][16][d], 16-byte aligned, n_pool_pages * Hkv * 16 <= 2^31 - 1
 * (the pools' extent: the kernel's copies never address past it);
 * page_table: int32 [ceil(T/16)], logical page -> physical page, every entry
 * in [0, n_pool_pages); n_splits: key-range partitions per KV head (1..256,
 * rounded up to a multiple of 8, the CTAs of one cluster; 0 = the engine's
 * choice); out: fp32 [Hq][d].  d in {64, 128}, Hq/Hkv <= 8, T >= 1.
 * Blocks until the kernel has finished (it reads the kernel's error word back):
 * a table entry outside [0, n_pool_pages) is replaced by page 0 on the device
 * and returns LLM_ERR_DEVICE (out then undefined); a page copy that never
 * lands within the kernel's 1 s bound returns LLM_ERR_TIMEOUT.  Other errors:
 * LLM_ERR_ARG (checked before any launch), LLM_ERR_CUDA.                      */
int llm_op_attention(const float *q, const void *k_pool, const void *v_pool,
                     const int32_t *page_table, int32_t n_pool_pages, int32_t T, int32_t Hq,
                     int32_t Hkv, int32_t d, int32_t n_splits, float *out, void *stream);

/* llm_op_attention without any device allocation.  There is no counterpart
 * in the source pages: this serves callers that may not allocate device memory
 * when they call in (a host framework that owns all device memory through its
 * own pool and forbids cudaMalloc on its threads, or latency-critical paths
 * where an allocation could lock or synchronise).  Same arguments, same kernel
 * and same result as llm_op_attention, but the scratch (per-split partials and
 * arrival counters) lives in a fixed 4 MiB array of device memory inside the
 * library, which every GPU that loads the library holds until exit.
 * Size limit: 256 + Hq * P * (d + 2) * 4 bytes <= 4 MiB, with P = n_splits (or
 * the engine's choice when 0), and Hkv <= 63; larger requests return
 * LLM_ERR_ARG before anything is launched.  Calls no cudaMalloc or cudaFree;
 * the counters are reset with cudaMemsetAsync on `stream` each call.  The
 * first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current, so make it before any
 * stream capture.  All calls on a device share the array: calls that may run
 * concurrently on the GPU (different streams without ordering) race.  Like
 * llm_op_attention it blocks until the kernel has finished and reports a bad
 * page (LLM_ERR_DEVICE) or a page wait that ran out (LLM_ERR_TIMEOUT).  The
 * array's address is looked up once per device and kept: do not use the
 * library across a cudaDeviceReset.                                           */
int llm_op_attention_noalloc(const float *q, const void *k_pool, const void *v_pool,
                             const int32_t *page_table, int32_t n_pool_pages, int32_t T,
                             int32_t Hq, int32_t Hkv, int32_t d, int32_t n_splits, float *out,
                             void *stream);

/* Weight dequantization for the batched prefill ("Bare-Metal LLM Inference on
 * NVIDIA H100", prefill path: dequantized tiles feed the tensor cores):
 * out[n][k] = fp16(code[n][k] * scale).  fmt 1 = INT4 group-128 (w: layout
 * LLM_LAYOUT_INT4_VALUESHUFFLE words [N][K/8], s: bf16 [N][K/128]; every INT4
 * weight is exact in fp16 while its scale is at least 2^-14), fmt 2 = INT8 per
 * row (w: int8 [N][K], s: fp32 [N]; rounded to nearest fp16).  out: fp16
 * [N][K], 16-byte aligned.  K % 128 == 0 (INT4) or K % 8 == 0 (INT8).       */
int llm_op_dequant_f16(int32_t fmt, const void *w, const void *s, int32_t N, int32_t K, void *out,
                       void *stream);

/* C[m][n] = sum_k A[m][k] * B[n][k] on the tcgen05 tensor cores: fp16 operands
 * staged by TMA, fp32 accumulation in tensor memory (the prefill GEMM).  A: fp16
 * [M][K], B: fp16 [N][K], both row-major and 16-byte aligned; C: fp32 [M][N].
 * M >= 1, N % 128 == 0, K % 64 == 0.  A wait inside the kernel that runs out
 * (1 s; only a stalled GPU) leaves C undefined.                               */
int llm_op_gemm_f16(const void *A, const void *B, int32_t M, int32_t N, int32_t K, float *C,
                    void *stream);

/* C[m][n] = sum_k A[m][k] * W[n][k] on the tcgen05 tensor cores with the
 * weights dequantized inside the kernel (the prefill GEMM as the engine runs
 * it): W is fmt 1 = INT4 group-128 (w: LLM_LAYOUT_INT4_VALUESHUFFLE words
 * [N][K/8], s: bf16 [N][K/128]) or fmt 2 = INT8 per row (w: int8 [N][K],
 * s: fp32 [N]); each code tile is converted to fp16 in tensor memory and
 * never written back (INT4: code x group scale, exact; INT8: the code, exact,
 * with the fp32 row scale applied to the fp32 sum).  A: fp16 [M][K],
 * C: fp32 [M][N], 16-byte aligned.  M >= 1, N % 128 == 0, K % 128 == 0.  The
 * result does not depend on the run (partial sums of a split K are added in a
 * fixed order).                                                              */
int llm_op_gemm_quant(int32_t fmt, const void *A, const void *w, const void *s, int32_t M, int32_t N,
                      int32_t K, float *C, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* QD_LLM_OPS_H */
