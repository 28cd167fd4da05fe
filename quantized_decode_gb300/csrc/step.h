// step.h - the persistent decode-step kernel: parameters shared by the host
// planner (engine.cu) and the kernel (k_step.cu).
//
// One launch runs the whole decode step: for every layer the phases
//   QKV  RMSNorm -> Q/K/V GEMV (+bias) -> per-head q/k norm + RoPE -> KV append
//   ATTN split-K GQA attention over the paged cache + log-sum-exp combine
//   O    o_proj GEMV + residual
//   GU   RMSNorm -> gate/up GEMV -> SiLU * mul
//   DOWN down GEMV + residual
// and then LM (final RMSNorm -> LM head GEMV -> argmax).  One CTA per SM; a
// phase waits for the phase it depends on through counters in device memory.
#pragma once

#include <cuda.h>

#include "kernels.h"

namespace qd {

constexpr int kStepSlotBytes = 9216;      // one ring item (1024-byte multiple: swizzled boxes)
constexpr int kStepResFloats = 2048;      // per-CTA row results of one phase
constexpr int kStepMaxSlots = 20;
constexpr int kStepProducers = 4;           // copy-issuing threads per CTA (one per producer warp)
// A GEMV ring item is kStepLines row-lines of one K-tile of up to
// kStepTileBytes bytes a row, loaded by one 3-D TMA box per matrix (rows x
// 128-byte chunks x 128 bytes, 128-byte swizzle: line i, chunk c sits in
// 128-byte segment i * chunks + c of the box with its 16-byte units
// XOR-permuted by the segment index), then (INT4) the 16-byte-aligned cover
// of the lines' whole scale rows at kStepScaleOff.  Gate/up items hold two
// boxes of two rows, the gate box at 0 and the up box at kStepUpOff (each box
// starts on a 1024-byte boundary), and two covers at kStepGuScaleOff and
// kStepGuScaleOff + kStepGuScaleSpan.
constexpr int kStepLines = 4;
constexpr int kStepTileBytes = 1792;
constexpr int kStepScaleOff = kStepLines * kStepTileBytes;
constexpr int kStepUpOff = 4096;
constexpr int kStepGuScaleOff = kStepUpOff + 2 * kStepTileBytes;
constexpr int kStepGuScaleSpan = 768;
// Staged activations: fp16 (INT4/INT8 weights) or bf16 hi/lo pairs (bf16
// weights) laid out as mma B fragments, then one fp32 correction per block.
constexpr int kStepMaxStageK = 18944;
constexpr int kStepStageBytes = kStepMaxStageK * 2 + 768 * 4;

enum StepPhase : int { kPhQkv = 0, kPhAttn = 1, kPhO = 2, kPhGu = 3, kPhDown = 4, kPhLm = 5, kPhCount = 6 };

// Step counters, per layer (zeroed by the last CTA of the step, so every step
// starts from zero).
constexpr int kSyncStride = 128;
constexpr int kSyncHeadsDone = 96;   // [0, Hq + 2 Hkv): rows arrived per head; 96: heads finished
constexpr int kSyncAttnCnt = 100;    // [100, 100 + Hkv): attention partials written per KV head
constexpr int kSyncAttnDone = 120;   // attention CTAs that wrote their combined slice
constexpr int kSyncODone = 121;      // CTAs past the o_proj epilogue
constexpr int kSyncGuDone = 122;
constexpr int kSyncDDone = 123;
constexpr int kSyncMaxHeads = 96;
constexpr int kSyncMaxKvHeads = 16;


// Weight tensor maps of a layer (3-D codes boxes, see above).
enum StepMap : int { kMapQ = 0, kMapK = 1, kMapV = 2, kMapO = 3, kMapGate = 4, kMapUp = 5, kMapDown = 6, kMapCount = 7 };

struct StepLayer {
    const CUtensorMap *tm;       // [kMapCount] in device memory
    const void *w[3], *s[3];     // q, k, v codes and scales
    const uint16_t *b[3];        // q, k, v bias (bf16) or null
    const void *wo, *so, *wg, *sg, *wu, *su, *wd, *sd;
    const uint16_t *attn_norm, *mlp_norm, *q_norm, *k_norm;
};

// One GEMV phase as the CTAs split it.
struct StepGeo {
    int fmt;        // kFmtInt4 / kFmtInt8 / kFmtBf16
    int N, K;       // output rows (GU: gate/up pairs) and inputs
    int row_bytes;  // bytes of one weight row
    int sr;         // INT4: bf16 scale bytes per row (K / 64); else 0
    int tk;         // bytes of one row in a K-tile (<= kStepTileBytes)
    int nt;         // K-tiles per row
    int bb;         // bytes of one mma block of a row: INT4 64 (128 codes), INT8 16, bf16 32
};

struct StepParams {
    CUtensorMap tm_k, tm_v;      // KV pools as 2-D [rows][d] bf16, 128-byte swizzled 16-row boxes
    CUtensorMap tm_lm;           // LM head codes (3-D box like the layer weights)
    StepGeo geo[kPhCount];
    const StepLayer *layers;     // [L], device memory
    int L, h, Hq, Hkv, d, F, V;
    float eps;
    const uint16_t *embed, *final_norm;
    const void *lm_w;
    const float *lm_scale;       // INT8 LM head row scales or null
    const int *page_table;
    int n_pages;
    const float2 *rope_cs;
    uint16_t *k_pool, *v_pool;   // all layers [L][pages][Hkv][16][d]
    DevState *st;
    float *x, *raw, *q, *attn, *u, *logits;
    float *part_o, *part_ml;     // attention partials [Hkv][P][G][d], [Hkv][P][G][2]
    float *lm_val;
    int *lm_idx;
    int *sync;                   // [L][kSyncStride] + 1 (LM arrival)
    int P;                       // attention splits per KV head (Hkv * P CTAs take part)
    int n_slots;                 // ring items
    int inflight;                // ring items a CTA may have in flight at once
    unsigned long long *prof;    // null, or 5 L + 2 phase timestamps (CTA 0)
    unsigned long long wait_ns;  // bound on every wait
    // Test hooks (llm_debug_step_wait): the phase-counter waits expect this many
    // arrivals more than will come and give up after counter_wait_ns; the
    // waits that guard copies in flight keep wait_ns.
    int test_extra_arrivals;
    unsigned long long counter_wait_ns;
};

// Host side (k_step.cu).
struct StepLaunch {
    const void *kernel = nullptr;
    int grid = 0, block = 0;
    size_t smem = 0;
};
// Chooses the instantiation and the launch shape; false if the model is outside
// what the persistent kernel supports (the engine then runs the kernel chain).
bool step_plan(StepParams &p, int weight_fmt, int lm_fmt, int n_sm, int max_smem, StepLaunch &out);
cudaError_t step_encode_kv_maps(StepParams &p, size_t total_rows);
// 3-D box map of a weight matrix [N][row_bytes] for phase geometry g (box:
// 128 bytes x g.tk / 128 chunks x `lines` rows); row_bytes % 128 == 0.
cudaError_t step_encode_weight_map(CUtensorMap *map, const void *w, int N, const StepGeo &g, int lines);
cudaError_t launch_step(const StepLaunch &sl, const StepParams &p, cudaStream_t stream);
// CTAs of the step kernel that fit on one SM (the launch needs >= 1).
cudaError_t step_occupancy(const StepLaunch &sl, int *blocks_per_sm);

}  // namespace qd
