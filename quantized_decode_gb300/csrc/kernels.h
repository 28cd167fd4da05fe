// kernels.h - launch interface of the decode-step kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qd {

constexpr int kPageTokens = 16;   // KV tokens per page (16-token pages, bf16)
constexpr int kGroup = 128;       // INT4 quantization group along K
constexpr int kMaxGqa = 8;        // query heads per KV head supported by the attention kernel
constexpr int kStatSlots = 256;   // (sum of squares, max) pairs per producer: one per CTA, >= grid
constexpr size_t kMaxSmemOptin = 227 * 1024;  // shared memory a CTA may opt in to (sm_103a)

// Byte ranges a kernel prefetches into L2 for a later kernel of the step
// (llm_set_l2_prefetch): every CTA issues bulk prefetches of its share of each
// range at its start, before its dependency wait.  Null ranges are skipped.
struct L2Range {
    const void *p;              // 16-byte aligned
    unsigned long long bytes;
};
constexpr int kMaxL2Ranges = 4;

// Device-side error word (sticky until the host clears it).
enum : int { kErrNone = 0, kErrBadPage = 1, kErrBadToken = 2, kErrBadPos = 3, kErrTimeout = 16 };

// kFmtInt4A8: INT4 g128 weights against activations quantized to int8 per
// 128-group inside the GEMV (dp4a), an opt-in decode variant.
enum WeightFormat : int { kFmtInt4 = 1, kFmtInt8 = 2, kFmtBf16 = 3, kFmtInt4A8 = 4 };

// Scalars of the running sequence, resident in device memory so that one
// captured graph serves every position.
struct DevState {
    int32_t pos;         // position the next step writes (= tokens in the cache)
    int32_t token;       // token the next step consumes
    int32_t last_token;  // argmax emitted by the most recent step
    int32_t err;         // sticky device error word (kErr*)
};

// Launch configuration shared by all kernels of one step.
struct LaunchCfg {
    cudaStream_t stream;
    bool pdl;     // programmatic dependent launch attribute
    int n_sm;     // SMs on the device
};

// RMSNorm -> Q/K/V GEMV (+bias) -> per-head (q/k RMSNorm) + RoPE -> q out,
// K/V appended to the paged cache at the current position.
struct QkvArgs {
    const void *w[3];       // q, k, v codes
    const void *s[3];       // q, k, v scales
    const uint16_t *b[3];   // q, k, v bias (bf16) or null
    int rows_q, rows_kv;    // Hq*d and Hkv*d
    int K;                  // hidden
    int d, Hq, Hkv;
    const float *x;         // residual [K] (ignored when embed != null)
    const long long *x2;    // the MLP's pending contribution (fixed point) added to x, or null; then no stats_in
    const uint16_t *embed;  // layer 0: bf16 embedding table [V][K]
    float *x_init;          // layer 0: residual initialised from the embedding row
    const uint16_t *gamma;  // attn_norm
    float eps;
    const uint16_t *q_gain, *k_gain;  // per-head RMSNorm gains, or null
    float *raw;             // [rows_q + 2 rows_kv] scratch
    float *q_out;           // [rows_q] rotated queries
    int *head_cnt;          // [Hq + 2 Hkv] completion counters (self-resetting)
    uint16_t *k_pool, *v_pool;  // this layer's pools [pages][Hkv][16][d]
    const int *page_table;
    int n_pages;
    const float2 *rope_cs;  // [max_context][d/2] (cos, sin)
    DevState *st;
    uint16_t *kv_new;       // [2][Hkv][d] bf16 copy of the appended K and V rows
    const float *stats_in;  // producer (ss, mx) pairs for x, or null (computed here)
    int ks;                 // set by the launcher: warps per tile along K
    unsigned long long *tl; // timeline slot of this launch, or null (TimelineMark)
    L2Range pf[kMaxL2Ranges];  // L2 prefetch for a later kernel, or all null
};

// y = W x with a fused epilogue: mode 0 stores (plus optional bias), mode 1
// adds into y (residual), mode 2 is the gate/up pair with SiLU*mul.
struct GemvArgs {
    int mode;
    const void *w, *s;      // codes and scales (gate for mode 2)
    const void *w2, *s2;    // up codes and scales (mode 2)
    const uint16_t *bias;   // mode 0 only
    int N, K;               // N output rows (mode 2: F hidden units)
    const float *x;         // input activations [K]
    const uint16_t *gamma;  // RMSNorm gain applied to x first, or null
    float eps;
    float *y;               // output [N]
    long long *fold;        // mode 1: y += fold (fixed point) and fold = 0 (fold_add), or fold = 0 only; or null
    int fold_add;
    const long long *x2;    // mode 2: a pending contribution (fixed point) added to x first, or null;
                            // then stats_in must be null (the statistics are computed here)
    const float *stats_in;  // producer (ss, mx) pairs for x, or null (computed here)
    float *stats_out;       // this kernel's (ss, mx) pairs for y, or null
    const uint16_t *stats_gamma;  // gain of y's consumer norm for mx (null: none)
    int ks;                 // set by the launcher: warps per tile along K
    unsigned long long *tl; // timeline slot of this launch, or null (TimelineMark)
    L2Range pf[kMaxL2Ranges];  // L2 prefetch for a later kernel, or all null
};

// The MLP block as one kernel (k_mlp.cu): RMSNorm -> gate/up -> SiLU * mul ->
// down, each CTA on a slice of the hidden units, D += its down partial sums.
struct MlpArgs {
    const void *wg, *sg, *wu, *su;  // gate / up codes and scales [F][h] (INT4: bf16 [F][h/128]; INT8: fp32 [F])
    const uint4 *wd;                // down codes, unit-major [F / C][h][16 B] (mlp_repack_down)
    const void *sd;                 // INT4: bf16 [F / 128][h] (repacked); INT8: fp32 [h] row scales
    int F, h;
    const float *x;                 // residual after the attention block [h]
    const uint16_t *gamma;          // mlp_norm
    float eps;
    const float *stats_in;          // o_proj's (ss, mx) pairs for x
    long long *D;                   // [h]: zero on entry; receives the block's output (fixed point, 2^-32)
    int prefetch_down;              // prefetch the CTA's down block into L2 at its start
    int *err;                       // device error word (kErrTimeout when a bounded copy wait runs out)
    unsigned long long wait_ns;     // bound on every wait of the kernel
    unsigned long long *tl;         // timeline slot of this launch, or null (TimelineMark)
};
bool mlp_shape_ok(int fmt, int h, int F);
cudaError_t launch_mlp(const LaunchCfg &lc, int fmt, const MlpArgs &a);
// Repack W_down [h][F] into the unit-major layout k_mlp reads (w_out: h * F / 2
// bytes INT4, h * F INT8; s_out: INT4 scales [F/128][h], unused for INT8).
cudaError_t mlp_repack_down(int fmt, const void *w, const void *s, int h, int F, void *w_out, void *s_out,
                            cudaStream_t stream);

// ---- multi-sequence decode (k_batch.cu) ----------------------------------------
// Y[b][n] = sum_k W[n][k] X[b][k] for b < B <= 8 sequences on the tensor cores
// (mma.sync, bf16 operands, fp32 accumulation), each weight read once.
struct BGemvArgs {
    int mode;                   // 0 store (+ bias), 1 add into y, 2 SiLU(gate) * up (w[0] gate, w2 up), 3 store
    int n_seg;                  // modes 0/1/3: stacked matrices w[0..n_seg) of seg_rows[i] rows (multiples of 16)
    const void *w[3], *s[3];    // codes (INT4 words / INT8 / bf16) and scales (INT4 bf16 [N][K/128], INT8 fp32 [N])
    const uint16_t *bias[3];    // mode 0: bf16 bias per segment, or null
    int seg_rows[3];
    const void *w2, *s2;        // mode 2: up codes and scales
    int N, K, B;                // N output rows (mode 2: hidden units), B sequences
    const float *x;             // [B][ldx] inputs
    int ldx;
    const uint16_t *gamma;      // RMSNorm gain applied to every input row first, or null
    float eps;
    float *y;                   // [B][ldy]
    int ldy;
    int ks;                     // set by the launcher: warps per tile along K
};
// Per (sequence, head): q/k RMSNorm, RoPE at the sequence's position, q out,
// K/V to slot pos % 16 of the sequence's page table[pos / 16]; sequences whose
// `part` flag is 0 are skipped.
struct BQkvPostArgs {
    const float *raw;           // [B][(Hq + 2 Hkv) d]
    int Hq, Hkv, d;
    const uint16_t *q_gain, *k_gain;
    float eps;
    const float2 *rope_cs;
    float *q_out;               // [B][Hq d]
    uint16_t *k_pool, *v_pool;  // this layer [pages][Hkv][16][d]
    const int *page_table;      // [B][max_pages]
    int max_pages, n_pages;
    DevState *st;               // [B]
    const int *part;            // [B] 1: the sequence takes part in this step
};
bool bgemv_shape_ok(int fmt, int N, int K, int mode);
cudaError_t launch_bgemv(const LaunchCfg &lc, int fmt, const BGemvArgs &a);
cudaError_t launch_bembed(cudaStream_t s, const uint16_t *embed, const DevState *st, int B, int h, float *x);
cudaError_t launch_bqkv_post(cudaStream_t s, const BQkvPostArgs &a, int B);
// pv, pi: [B][32] scratch of the split argmax.
cudaError_t launch_bargmax(cudaStream_t s, const float *logits, int V, DevState *st, int B, const int *part,
                           float *pv, int *pi);

// Final RMSNorm -> LM head GEMV -> logits + greedy argmax (lowest index on
// ties).  The last CTA reduces the per-CTA maxima, writes the token into the
// state (as the next step's input) and advances the position when `advance`.
struct LmHeadArgs {
    int fmt;                // kFmtBf16 or kFmtInt8
    const void *w;          // bf16 [V][K] or int8 [V][K]
    const float *scale;     // int8 row scales or null
    const uint16_t *gamma;
    float eps;
    int N, K;
    const float *x;
    const long long *x2;    // the MLP's pending contribution (fixed point) added to x, or null; then no stats_in
    float *logits;          // [N]
    float *part_val;        // [grid] per-CTA maxima
    int *part_idx;          // [grid]
    int *counter;           // self-resetting
    int *token_out;         // where the argmax goes (state or user buffer)
    DevState *st;           // non-null: last_token/token written, pos advanced
    int advance;
    const float *stats_in;  // producer (ss, mx) pairs for x, or null (computed here)
    unsigned long long *tl; // timeline slot of this launch, or null (TimelineMark)
};

// Temperature / top-k / top-p sampling of the next token from the logits (in
// place of the greedy argmax).  One CTA; the token to token_out and, with a
// state, into it as the next step's input (pos advanced when `advance`); the
// draw's counter is st->pos (or `counter` without a state).
constexpr int kMaxTopK = 1024;
struct SampleArgs {
    const float *logits;    // [V]
    int V;
    float temperature;      // > 0
    int top_k;              // 1 .. min(V, kMaxTopK)
    float top_p;            // (0, 1]
    uint64_t seed;
    uint64_t counter;       // without a state
    int *token_out;
    DevState *st;           // or null
    int advance;
    unsigned long long *tl; // timeline slot of this launch, or null (TimelineMark)
};
cudaError_t launch_sample(const LaunchCfg &lc, const SampleArgs &a);

// Split-K decode attention over the paged cache with the LSE combine.
struct AttnArgs {
    const float *q;                    // [Hq][d] rotated
    const uint16_t *k_pool, *v_pool;   // this layer [pages][Hkv][16][d]
    const int *page_table;
    int n_pages;
    const DevState *st;                // T = st->pos + 1 when T_fixed < 0
    int T_fixed;
    int Hq, Hkv, d, P;                 // P = splits per KV head
    float *part_o;                     // [Hkv][P][G][d]
    float *part_ml;                    // [Hkv][P][G][2]
    int *counter;                      // [Hkv] self-resetting
    float *out;                        // [Hq][d]
    int *err;
    const uint16_t *kv_new;            // [2][Hkv][d] appended K/V row, or null (all rows in pages)
    int cs;                            // CTAs per cluster: 8 (0 = 8), 16 (d = 128 only) or 4
    CUtensorMap k_map, v_map;          // set by the launcher: the pools as 2-D tensors
                                       // [pages * Hkv * 16][d] for TMA page loads
    float *stats_out;                  // (ss, mx) pairs of out, or null: slot g per KV head, or with
                                       // one 16-CTA cluster per head slot 16 g + rank (others untouched)
    unsigned long long *tl; // timeline slot of this launch, or null (TimelineMark)
    // o_proj folded in (one cluster per KV head only, INT4 W_o, d = 128; see AttnFold), in
    // device memory; out is then not written.  Null: no fold.
    const struct AttnFold *fold;
};

// The o_proj fold of one layer: the cluster of KV head g multiplies its G*d outputs by
// W_o's columns [g G d, (g + 1) G d) and adds the rows to out (fixed point, 2^-32), CTA r
// of the cluster taking rows [r hidden / cs, (r + 1) hidden / cs).
struct AttnFold {
    CUtensorMap wo_map;                // W_o as 32-bit words [hidden][Hq d / 8], boxes of G d / 8 words
                                       // x hidden / cs rows
    const uint16_t *so;                // bf16 scales [hidden][Hq d / 128]
    long long *out;                    // [hidden]
    int hidden;
};


// Each launcher returns the launch's cudaError_t.
cudaError_t launch_qkv(const LaunchCfg &lc, int fmt, const QkvArgs &a);
cudaError_t launch_gemv(const LaunchCfg &lc, int fmt, const GemvArgs &a);
cudaError_t launch_lm_head(const LaunchCfg &lc, const LmHeadArgs &a, int grid);
cudaError_t launch_attention(const LaunchCfg &lc, const AttnArgs &a);
// The TMA maps of a's pools (boxes of 64 columns x 16 rows, 128-byte swizzle).
cudaError_t attention_pool_maps(AttnArgs &a);

// Grid sizes and shape checks used by the engine when it plans buffers.
int lm_head_grid(const LaunchCfg &lc, int N);
// Splits per KV head: as many 8-CTA clusters as fill the SMs and are resident
// at once on this device (cudaOccupancyMaxActiveClusters).
int default_splits(int n_sm, int Hq, int Hkv, int d, int max_pages);
// The engine's attention shape: P splits per KV head in clusters of cs CTAs.
struct AttnPlan {
    int P, cs;
};
AttnPlan plan_attention(int n_sm, int Hq, int Hkv, int d, int max_pages);
// Whether attention with plan `ap` can fold o_proj in (shapes and shared memory).
bool attn_fold_ok(int fmt, int Hq, int Hkv, int d, int hidden, const AttnPlan &ap);
// The fold of one layer (host copy, to be copied to device memory): W_o codes (16-byte
// aligned) and scales, the output buffer.
cudaError_t attn_fold_args(AttnFold &f, const void *wo, const uint16_t *so, long long *out, int Hq, int Hkv, int d,
                           int hidden, const AttnPlan &ap);

// QKV projection + attention of a layer in one kernel (one 16-CTA cluster per
// KV head; models without q/k norms, d = 128).  `at` as for launch_attention
// with P = cs = 16 and out set; qa as for launch_qkv (q_out, raw, head_cnt and
// kv_new unused).
bool qkv_attn_fusable(int fmt, int Hq, int Hkv, int d, int K, bool qk_norm, const AttnPlan &plan);
cudaError_t launch_qkv_attn(const LaunchCfg &lc, int fmt, const QkvArgs &qa, const AttnArgs &at);
int attention_split_multiple();  // split counts are multiples of the attention cluster size
bool gemv_shape_ok(int fmt, int N, int K, int mode);
bool qkv_shape_ok(int fmt, int rows_q, int rows_kv, int K, int d);
bool lm_head_shape_ok(int fmt, int N, int K);

}  // namespace qd
