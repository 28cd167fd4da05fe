// prefill.h - launch interface of the prompt (prefill) kernels (host side).
//
// Prefill runs the decode step's math for n prompt tokens at once: the
// linear layers become GEMMs on the tcgen05 tensor cores (weights dequantized
// to fp16 tiles, activations fp16, fp32 accumulators in TMEM), attention is
// causal over the prompt plus whatever the cache already holds, and only the
// last row goes through the LM head.
#pragma once

#include <cuda.h>

#include "kernels.h"

namespace qd {

// ---- tcgen05 GEMM: D[M][N] = A[M][K] * B[N][K]^T (fp16 in, fp32 accumulate) ----
constexpr int kTcBM = 128, kTcBN = 128, kTcBK = 64;

enum TcEpilogue : int {
    kEpiStore = 0,   // C[m][n] = D
    kEpiAdd = 1,     // C[m][n] += D (residual)
    kEpiSwiGlu = 2,  // B rows interleaved per 128-row tile as 64 gate rows then the
                     // matching 64 up rows: H[m][n/2 + j] = fp16(silu(gate_j) * up_j)
};

struct TcGemmArgs {
    int M, N, K;            // N % 128 == 0, K % 64 == 0, M >= 1 (A rows past M read as zero)
    int mode;               // TcEpilogue
    float *c;               // kEpiStore / kEpiAdd: fp32 [M][ldc]
    int ldc;
    uint16_t *h;            // kEpiSwiGlu: fp16 [M][ldh]
    int ldh;
    int *err;               // device error word (kErrTimeout on a wait that ran out), or null
    unsigned long long wait_ns;  // bound on every wait of the kernel
};

// Tensor map of a row-major fp16 matrix [rows][cols] for the GEMM's operand
// tiles (128 rows x 64 columns, 128-byte swizzle).  cols % 64 == 0, base
// 16-byte aligned.
cudaError_t tc_operand_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols);
cudaError_t launch_tc_gemm(cudaStream_t stream, const CUtensorMap &a_map, const CUtensorMap &b_map,
                           const TcGemmArgs &a);

// ---- the same GEMM with quantized weights dequantized inside the kernel -------
// B = the weight codes: up to three stacked matrices (QKV: seg_rows = q, k, v
// rows, each a multiple of 128), or (interleave) a gate/up pair of seg_rows[0]
// rows each, whose 128-row tiles hold 64 gate rows then the matching 64 up rows.
// The kernel computes 128 weight rows x 256 prompt rows per CTA with the
// dequantized weights in tensor memory; when that leaves most SMs idle it
// splits K over a cluster of 2 or 4 CTAs and adds their partial sums in a
// fixed order (results do not depend on the run).
struct TcQuantB {
    int fmt;                 // kFmtInt4 (bf16 group scales) / kFmtInt8 (fp32 row scales)
    int interleave;
    int n_seg;
    int seg_rows[3];
    const void *scale[3];
};
// Tensor map of a code matrix [rows][K] (INT4: K/2 bytes a row) for tiles of
// box_rows (128, or 64 for an interleaved pair) x 64 codes.
cudaError_t tc_weight_map(CUtensorMap *map, const void *codes, int fmt, uint64_t rows, uint64_t K, int box_rows);
// Tensor map of the activations A [rows][cols] fp16 of the quantized GEMM
// (tiles of 256 rows x 64 columns, 128-byte swizzle; rows past `rows` read as
// zero).  cols % 64 == 0, base 16-byte aligned.
cudaError_t tc_act_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols);
// a_map from tc_act_map, w_maps from tc_weight_map.  kEpiSwiGlu needs interleave.
// With pdl the launch may overlap the previous kernel of the stream: only the
// weight codes are read before the kernel waits for it.
cudaError_t launch_tc_gemm_q(cudaStream_t stream, const CUtensorMap &a_map, const CUtensorMap (&w_maps)[3],
                             const TcQuantB &b, const TcGemmArgs &a, bool pdl = false);
// K split of a launch (1, 2 or 4) on a device with n_sm SMs.
int tc_gemm_q_split(int M, int N, int K, int mode, int n_sm);

// ---- weight dequantization to fp16 rows ----------------------------------------
// out[r][k] = code[src(r)][k] * scale (INT4: bf16 group scale; INT8: fp32 row
// scale), fp16.  With `interleave` (gate/up pair, w2/s2 = up matrix) output
// tile t of 128 rows holds gate rows [64t, 64t + 64) then up rows [64t, 64t + 64).
struct DequantArgs {
    int fmt;                 // kFmtInt4 / kFmtInt8
    const void *w, *s;       // codes and scales
    const void *w2, *s2;     // second matrix (interleave) or null
    int N, K;                // rows of one matrix, K % 128 == 0 (INT4) / K % 16 == 0 (INT8)
    uint16_t *out;           // fp16 [N (x2 when interleaved)][K]
};
cudaError_t launch_dequant(cudaStream_t stream, int n_sm, const DequantArgs &a);

// ---- row kernels -----------------------------------------------------------------
// x[i] = float(E[tok[i]]) for the n prompt rows.
cudaError_t launch_embed_rows(cudaStream_t stream, const uint16_t *embed, const int *tokens, int n, int h,
                              float *x);
// out[i] = fp16(x[i] / rms(x[i]) * gamma) for n rows of width h.
cudaError_t launch_rmsnorm_rows(cudaStream_t stream, const float *x, const uint16_t *gamma, float eps, int n,
                                int h, uint16_t *out);

// QKV post-processing for n rows at positions pos0 .. pos0+n-1: bias, optional
// per-head q/k RMSNorm, RoPE; K and V rounded to bf16 into the paged pools,
// queries kept as bf16 hi/lo pairs for the attention kernel.
struct QkvRowsArgs {
    const float *raw;        // [n][(Hq + 2 Hkv) d] GEMM output
    const uint16_t *bq, *bk, *bv;      // bf16 bias or null
    const uint16_t *q_gain, *k_gain;   // bf16 per-head RMSNorm gains or null
    float eps;
    int n, pos0, Hq, Hkv, d;
    const float2 *rope_cs;   // [max_context][d/2]
    uint16_t *k_pool, *v_pool;         // this layer [pages][Hkv][16][d]
    const int *page_table;
    int n_pages;
    uint16_t *q_hi, *q_lo;   // bf16 [n][Hq][d]
    int *err;
};
cudaError_t launch_qkv_rows(cudaStream_t stream, const QkvRowsArgs &a);

// Causal GQA attention of n query rows (positions pos0 .. pos0+n-1) over the
// paged cache (keys 0 .. pos): out fp16 [n][Hq][d].
struct AttnRowsArgs {
    const uint16_t *q_hi, *q_lo;       // bf16 [n][Hq][d]
    const uint16_t *k_pool, *v_pool;   // this layer
    const int *page_table;
    int n_pages;
    int n, pos0, Hq, Hkv, d;
    uint16_t *out;                      // fp16 [n][Hq * d]
    int *err;
};
cudaError_t launch_attn_rows(cudaStream_t stream, const AttnRowsArgs &a);

}  // namespace qd
