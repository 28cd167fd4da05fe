// engine.cu - the decode engine behind llm.h: validation, HBM layout, the step
// plan, single-graph capture and the host/device handshake per step.
//
// One decode step = for each layer [QKV+RoPE+append] -> [split-K attention +
// combine] -> [o_proj + residual] -> [RMSNorm + gate/up + SiLU*mul] ->
// [down + residual], then [final RMSNorm + LM head + argmax].  By default the
// step is a chain of 5L + 1 kernels; on request (llm_set_persistent) it is one
// persistent kernel (k_step.cu: one CTA per SM, weights streamed by TMA
// through a shared-memory ring, phases ordered by device counters).  Either
// form is captured once into a CUDA graph.  Position and input token live in
// device memory (DevState), so the same graph replays at every position ("How
// To Construct Your Personal LLM Runtime From Scratch", §6); the page for
// position pos is page_table[pos/16], read on the device, so no host-side
// branch on page boundaries is needed.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/llm.h"
#include "kernels.h"
#include "prefill.h"
#include "step.h"

using namespace qd;

// llm_set_l2_prefetch flags (see llm.h)
enum : int {
    kL2pfQkvMlp = 1,    // QKV prefetches the layer's gate and up weights
    kL2pfGuDown = 2,    // gate/up prefetches the layer's down weights
    kL2pfDownNext = 4,  // down prefetches the next layer's QKV and o_proj codes
    kL2pfQkvO = 8,      // QKV prefetches the layer's o_proj weights (when bit 1 is clear)
    kL2pfOMlp = 16,     // o_proj prefetches the layer's gate and up weights
    kL2pfAll = 31
};

struct llm_t {
    llm_config cfg;
    void *weight_buffer = nullptr;  // llm_create_from_file: the weights' device copy, owned
    int fmt = 0;
    std::vector<llm_layer_weights> layers;
    llm_weights w{};
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    int device = 0;
    LaunchCfg lc{};

    uint16_t *k_pool = nullptr, *v_pool = nullptr;
    size_t layer_kv_elems = 0;
    int *page_table = nullptr;
    int n_pages = 0;
    float2 *rope_cs = nullptr;
    DevState *st = nullptr;
    float *x = nullptr, *raw = nullptr, *q = nullptr, *attn = nullptr, *u = nullptr, *logits = nullptr;
    int *head_cnt = nullptr, *attn_cnt = nullptr, *lm_counter = nullptr, *lm_part_idx = nullptr;
    float *part_o = nullptr, *part_ml = nullptr, *lm_part_val = nullptr;
    float *stats = nullptr;     // 4 x kStatSlots (ss, mx) pairs: attention, o_proj, gate/up, down outputs
    uint16_t *kv_new = nullptr; // [2][Hkv][d] appended rows of the current step
    int P = 1, attn_cs = 8, lm_grid = 1;
    // llm_set_sampling: temperature / top-k / top-p instead of the greedy argmax
    bool sampling = false;
    bool act_int8 = false;      // llm_set_act_int8: o_proj, gate/up, down on int8 activations
    float samp_t = 0.f, samp_p = 1.f;
    int samp_k = 1;
    uint64_t samp_seed = 0;
    int *samp_scratch = nullptr;  // the LM head's unused argmax while sampling
    int l2pf = 0;               // llm_set_l2_prefetch flags
    // the MLP block as one kernel (k_mlp.cu): repacked down weights per layer and the
    // buffer D of the block's pending contribution to the residual
    bool mlp_ok = false;        // the model's shapes fit it
    bool mlp_fused = false;     // llm_set_fused_mlp (on by default where it fits)
    char *mlp_buf = nullptr;    // repacked down codes (+ INT4 scales) of every layer
    size_t mlp_w_bytes = 0, mlp_s_bytes = 0;  // per layer
    long long *mlp_d = nullptr;  // fixed point, 2^-32 units
    long long *o_d = nullptr;    // o_proj folded into the attention: its pending output (fixed point)
    AttnFold *o_fold_args = nullptr;  // per layer, device memory
    bool o_fold_ok = false;      // the attention plan and shapes allow the fold
    bool o_fold = false;         // llm_set_o_fold
    std::vector<int32_t> kinds; // kind of every launch of the captured step (llm_step_kinds)
    bool fused_ok = false;      // the model fits the fused QKV + attention kernel
    bool fused = false;         // llm_set_fused_attention

    // persistent whole-step kernel
    bool step_ok = false;       // the model fits the persistent kernel
    bool persistent = false;    // the step runs as the persistent kernel
    StepParams sp{};
    StepLaunch sl{};
    StepLayer *d_layers = nullptr;
    CUtensorMap *d_maps = nullptr;  // [n_layers][kMapCount] weight boxes of the persistent kernel
    int *step_sync = nullptr;
    unsigned long long *prof = nullptr;

    // batched prefill (tcgen05 GEMMs); buffers allocated by the first call
    bool pf_ok = false;         // the model's shapes fit the GEMM path
    bool pf_batched = true;     // llm_set_prefill_batched
    bool pf_ready = false;
    int pf_rows = 0;            // prompt rows per chunk
    float *pf_x = nullptr, *pf_raw = nullptr;
    uint16_t *pf_a = nullptr, *pf_u = nullptr, *pf_qh = nullptr, *pf_ql = nullptr;
    int *pf_tok = nullptr;
    CUtensorMap pf_map_ah{}, pf_map_aq{}, pf_map_u{};
    std::vector<CUtensorMap> pf_wmaps;  // per layer: q, k, v, o, gate, up, down code tiles

    int32_t *pinned = nullptr;  // host staging: [0] forced token, [2..3] last_token, err
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    bool use_graph = true;
    int32_t seq_len = 0;
    bool have_token = false;
    bool stepped = false;
};

namespace {

__global__ void k_set_state(DevState *st, int token, int pos, int clear_err) {
    if (token >= 0) st->token = token;
    if (pos >= 0) st->pos = pos;
    if (clear_err) st->err = 0;
}

bool aligned16(const void *p) { return p && ((uintptr_t)p & 15) == 0; }

template <typename T>
cudaError_t dalloc(T **p, size_t count) {
    return cudaMalloc(reinterpret_cast<void **>(p), count * sizeof(T));
}

void free_all(llm_t *h) {
    if (h->exec) cudaGraphExecDestroy(h->exec);
    if (h->graph) cudaGraphDestroy(h->graph);
    void *bufs[] = {h->k_pool, h->v_pool, h->page_table, h->rope_cs, h->st, h->x, h->raw, h->q,
                    h->attn, h->u, h->logits, h->head_cnt, h->attn_cnt, h->lm_counter,
                    h->lm_part_idx, h->part_o, h->part_ml, h->lm_part_val, h->stats, h->kv_new,
                    h->d_layers, h->d_maps, h->step_sync, h->prof, h->pf_x, h->pf_raw, h->pf_a, h->pf_u,
                    h->pf_qh, h->pf_ql, h->pf_tok, h->samp_scratch, h->mlp_buf, h->mlp_d, h->o_d,
                    h->o_fold_args};
    for (void *b : bufs)
        if (b) cudaFree(b);
    if (h->pinned) cudaFreeHost(h->pinned);
    if (h->own_stream && h->stream) cudaStreamDestroy(h->stream);
}

int validate(const llm_config *c, const llm_weights *w) {
    if (!c || !w || !w->layers) return LLM_ERR_ARG;
    if (c->weight_format == LLM_FMT_INT4_G128) {
        if (c->layout_id != LLM_LAYOUT_INT4_VALUESHUFFLE) return LLM_ERR_LAYOUT;
    } else if (c->weight_format == LLM_FMT_INT8_ROW) {
        if (c->layout_id != LLM_LAYOUT_INT8_ROW) return LLM_ERR_LAYOUT;
    } else {
        return LLM_ERR_ARG;
    }
    if (c->n_layers < 1 || c->hidden < 1 || c->n_q_heads < 1 || c->n_kv_heads < 1 || c->mlp < 1 ||
        c->vocab < 1 || c->max_context < 1)
        return LLM_ERR_ARG;
    if (c->page_tokens != kPageTokens || c->vocab % 64 != 0) return LLM_ERR_ARG;
    if (c->head_dim != 64 && c->head_dim != 128) return LLM_ERR_ARG;
    if (c->n_q_heads % c->n_kv_heads != 0 || c->n_q_heads / c->n_kv_heads > kMaxGqa) return LLM_ERR_ARG;
    if (!(c->rms_eps >= 0.f) || !(c->rope_base > 0.f)) return LLM_ERR_ARG;
    const int fmt = c->weight_format == LLM_FMT_INT4_G128 ? kFmtInt4 : kFmtInt8;
    const int h = c->hidden, d = c->head_dim, rq = c->n_q_heads * d, rkv = c->n_kv_heads * d;
    if (!qkv_shape_ok(fmt, rq, rkv, h, d)) return LLM_ERR_ARG;
    if (!gemv_shape_ok(fmt, h, rq, 1) || !gemv_shape_ok(fmt, c->mlp, h, 2) ||
        !gemv_shape_ok(fmt, h, c->mlp, 1))
        return LLM_ERR_ARG;
    const int lm_fmt = fmt == kFmtInt8 && !c->tied_lm_head ? kFmtInt8 : kFmtBf16;
    if (!lm_head_shape_ok(lm_fmt, c->vocab, h)) return LLM_ERR_ARG;
    if (!aligned16(w->embed) || !aligned16(w->final_norm)) return LLM_ERR_ARG;
    if (!c->tied_lm_head) {
        if (!aligned16(w->lm_head)) return LLM_ERR_ARG;
        if (fmt == kFmtInt8 && !aligned16(w->lm_scale)) return LLM_ERR_ARG;
    }
    for (int l = 0; l < c->n_layers; ++l) {
        const llm_layer_weights &L = w->layers[l];
        const void *req[] = {L.wq, L.sq, L.wk, L.sk, L.wv, L.sv, L.wo, L.so, L.wg, L.sg,
                             L.wu, L.su, L.wd, L.sd, L.attn_norm, L.mlp_norm};
        for (const void *p : req)
            if (!aligned16(p)) return LLM_ERR_ARG;
        if (c->qkv_bias && (!L.bq || !L.bk || !L.bv)) return LLM_ERR_ARG;
        if (c->qk_norm && (!aligned16(L.q_norm) || !aligned16(L.k_norm))) return LLM_ERR_ARG;
    }
    return LLM_OK;
}

}  // namespace

// The single-sequence engine's checks of a configuration and its weights, shared
// with the multi-sequence engine (batch.cu).
int engine_validate(const llm_config *c, const llm_weights *w) { return validate(c, w); }

namespace {

// The sampler after the LM head: the token into the state (the next step's
// input), the position advanced; the draw's counter is the sampled position.
SampleArgs sampler_args(const llm_t *h) {
    SampleArgs sa{};
    sa.logits = h->logits; sa.V = h->cfg.vocab;
    sa.temperature = h->samp_t; sa.top_k = h->samp_k; sa.top_p = h->samp_p; sa.seed = h->samp_seed;
    sa.token_out = &h->st->last_token; sa.st = h->st; sa.advance = 1;
    return sa;
}

// Bytes of one packed weight matrix [N][K] and of its scales.
size_t code_bytes(const llm_t *h, int N, int K) { return h->fmt == kFmtInt4 ? (size_t)N * K / 2 : (size_t)N * K; }
size_t scale_bytes(const llm_t *h, int N, int K) {
    return h->fmt == kFmtInt4 ? (size_t)N * (K / kGroup) * 2 : (size_t)N * 4;
}

// Enqueue one whole decode step (5L + 1 kernels).  With `ev`, event k is
// recorded before kernel k and event 5L+1 after the last one.
// Format of the o_proj, gate/up and down GEMVs (INT4 models may run them on int8 activations).
int gemv_fmt(const llm_t *h) { return h->act_int8 ? kFmtInt4A8 : h->fmt; }

// With `tl`, launch i of the step carries timestamp slot tl[i] (TimelineMark);
// *n_launch receives the number of kernels the step launched.
cudaError_t enqueue_step(llm_t *h, cudaEvent_t *ev = nullptr, unsigned long long *tl = nullptr,
                         int *n_launch = nullptr) {
    if (h->persistent && !ev) return launch_step(h->sl, h->sp, h->stream);
    const llm_config &c = h->cfg;
    const int d = c.head_dim, rq = c.n_q_heads * d, rkv = c.n_kv_heads * d;
    cudaError_t e;
    int k = 0;
    int kl = 0;
    h->kinds.clear();
    // timestamp slot of the next launch, which is of kind `kind` (LLM_KIND_*)
    auto slot = [&](int kind) -> unsigned long long * {
        unsigned long long *p = tl ? tl + kl : nullptr;
        ++kl;
        h->kinds.push_back(kind);
        return p;
    };
    const bool fmlp = h->mlp_fused && !h->act_int8;  // int8 activations keep the separate GEMVs
    // o_proj inside the attention clusters: its rows land in o_d, which gate/up adds to x
    // (computing its RMSNorm statistics itself) and down folds into the residual and zeroes
    const bool ofold = h->o_fold && !fmlp && !h->fused && !h->act_int8;
    float *st_attn = h->stats, *st_o = h->stats + 2 * kStatSlots;
    float *st_gu = h->stats + 4 * kStatSlots, *st_down = h->stats + 6 * kStatSlots;
    auto mark = [&]() -> cudaError_t { return ev ? cudaEventRecord(ev[k++], h->stream) : cudaSuccess; };
    for (int l = 0; l < c.n_layers; ++l) {
        const llm_layer_weights &L = h->layers[l];
        QkvArgs qa{};
        qa.w[0] = L.wq; qa.w[1] = L.wk; qa.w[2] = L.wv;
        qa.s[0] = L.sq; qa.s[1] = L.sk; qa.s[2] = L.sv;
        if (c.qkv_bias) {
            qa.b[0] = (const uint16_t *)L.bq;
            qa.b[1] = (const uint16_t *)L.bk;
            qa.b[2] = (const uint16_t *)L.bv;
        }
        qa.rows_q = rq; qa.rows_kv = rkv; qa.K = c.hidden; qa.d = d;
        qa.Hq = c.n_q_heads; qa.Hkv = c.n_kv_heads;
        qa.x = h->x;
        qa.x2 = fmlp && l > 0 ? h->mlp_d : nullptr;  // the previous layer's MLP output is still in D
        qa.embed = l == 0 ? (const uint16_t *)h->w.embed : nullptr;
        qa.x_init = h->x;
        qa.gamma = (const uint16_t *)L.attn_norm;
        qa.eps = c.rms_eps;
        if (c.qk_norm) {
            qa.q_gain = (const uint16_t *)L.q_norm;
            qa.k_gain = (const uint16_t *)L.k_norm;
        }
        qa.raw = h->raw; qa.q_out = h->q; qa.head_cnt = h->head_cnt;
        qa.k_pool = h->k_pool + (size_t)l * h->layer_kv_elems;
        qa.v_pool = h->v_pool + (size_t)l * h->layer_kv_elems;
        qa.page_table = h->page_table; qa.n_pages = h->n_pages;
        qa.rope_cs = h->rope_cs; qa.st = h->st;
        qa.kv_new = h->kv_new; qa.stats_in = l == 0 || fmlp ? nullptr : st_down;
        {
            int n = 0;
            if (h->l2pf & kL2pfQkvMlp) {  // gate and up of this layer, during the attention block
                qa.pf[n++] = {L.wg, code_bytes(h, c.mlp, c.hidden)};
                qa.pf[n++] = {L.wu, code_bytes(h, c.mlp, c.hidden)};
                qa.pf[n++] = {L.sg, scale_bytes(h, c.mlp, c.hidden)};
                qa.pf[n++] = {L.su, scale_bytes(h, c.mlp, c.hidden)};
            } else if (h->l2pf & kL2pfQkvO) {
                qa.pf[n++] = {L.wo, code_bytes(h, c.hidden, rq)};
                qa.pf[n++] = {L.so, scale_bytes(h, c.hidden, rq)};
            }
        }

        AttnArgs aa{};
        aa.q = h->q; aa.k_pool = qa.k_pool; aa.v_pool = qa.v_pool;
        aa.page_table = h->page_table; aa.n_pages = h->n_pages;
        aa.st = h->st; aa.T_fixed = -1;
        aa.Hq = c.n_q_heads; aa.Hkv = c.n_kv_heads; aa.d = d; aa.P = h->P; aa.cs = h->attn_cs;
        aa.part_o = h->part_o; aa.part_ml = h->part_ml; aa.counter = h->attn_cnt;
        aa.out = h->attn; aa.err = &h->st->err;
        aa.kv_new = h->kv_new; aa.stats_out = st_attn;
        if (ofold) {
            aa.fold = h->o_fold_args + l;
            aa.stats_out = nullptr;
        }
        // The step's first kernel reads the position before its dependency wait,
        // so it starts only after the previous step has ended (no early launch).
        LaunchCfg lc = h->lc;
        if (l == 0) lc.pdl = false;
        if (h->fused) {
            qa.tl = slot(LLM_KIND_QKV_ATTENTION);
            if ((e = mark()) != cudaSuccess || (e = launch_qkv_attn(lc, h->fmt, qa, aa)) != cudaSuccess ||
                (e = mark()) != cudaSuccess)
                return e;
        } else {
            qa.tl = slot(LLM_KIND_QKV);
            aa.tl = slot(LLM_KIND_ATTENTION);
            if ((e = mark()) != cudaSuccess || (e = launch_qkv(lc, h->fmt, qa)) != cudaSuccess) return e;
            if ((e = mark()) != cudaSuccess || (e = launch_attention(h->lc, aa)) != cudaSuccess) return e;
        }

        GemvArgs o{};
        o.mode = 1; o.w = L.wo; o.s = L.so; o.N = c.hidden; o.K = rq; o.x = h->attn; o.y = h->x;
        if (h->l2pf & kL2pfOMlp) {  // gate and up of this layer
            o.pf[0] = {L.wg, code_bytes(h, c.mlp, c.hidden)};
            o.pf[1] = {L.wu, code_bytes(h, c.mlp, c.hidden)};
            o.pf[2] = {L.sg, scale_bytes(h, c.mlp, c.hidden)};
            o.pf[3] = {L.su, scale_bytes(h, c.mlp, c.hidden)};
        }
        o.stats_in = st_attn; o.stats_out = st_o; o.stats_gamma = (const uint16_t *)L.mlp_norm;
        if (fmlp) {  // fold the previous layer's D into x (a new step starts from the embedding: zero only)
            o.fold = h->mlp_d;
            o.fold_add = l > 0;
        }
        if (ofold) {
            if ((e = mark()) != cudaSuccess) return e;  // the o_proj region of llm_profile_step: empty
        } else {
            o.tl = slot(LLM_KIND_O_PROJ);
            if ((e = mark()) != cudaSuccess || (e = launch_gemv(h->lc, gemv_fmt(h), o)) != cudaSuccess) return e;
        }

        if (fmlp) {
            MlpArgs m{};
            m.wg = L.wg; m.sg = L.sg; m.wu = L.wu; m.su = L.su;
            m.wd = reinterpret_cast<const uint4 *>(h->mlp_buf + (size_t)l * (h->mlp_w_bytes + h->mlp_s_bytes));
            m.sd = h->fmt == kFmtInt4 ? (const void *)(h->mlp_buf + (size_t)l * (h->mlp_w_bytes + h->mlp_s_bytes) +
                                                       h->mlp_w_bytes)
                                      : L.sd;
            m.F = c.mlp; m.h = c.hidden; m.x = h->x; m.gamma = (const uint16_t *)L.mlp_norm; m.eps = c.rms_eps;
            m.stats_in = st_o; m.D = h->mlp_d; m.prefetch_down = 1;
            m.err = &h->st->err; m.wait_ns = 1000000000ull;
            m.tl = slot(LLM_KIND_MLP);
            // the gate/up and down regions of llm_profile_step: the kernel, then nothing
            if ((e = mark()) != cudaSuccess || (e = launch_mlp(h->lc, h->fmt, m)) != cudaSuccess ||
                (e = mark()) != cudaSuccess)
                return e;
            continue;
        }

        GemvArgs gu{};
        gu.mode = 2; gu.w = L.wg; gu.s = L.sg; gu.w2 = L.wu; gu.s2 = L.su;
        gu.N = c.mlp; gu.K = c.hidden; gu.x = h->x;
        gu.gamma = (const uint16_t *)L.mlp_norm; gu.eps = c.rms_eps; gu.y = h->u;
        gu.stats_in = ofold ? nullptr : st_o; gu.stats_out = st_gu;
        gu.x2 = ofold ? h->o_d : nullptr;
        gu.tl = slot(LLM_KIND_GATE_UP);
        if (h->l2pf & kL2pfGuDown) {  // down of this layer
            gu.pf[0] = {L.wd, code_bytes(h, c.hidden, c.mlp)};
            gu.pf[1] = {L.sd, scale_bytes(h, c.hidden, c.mlp)};
        }
        if ((e = mark()) != cudaSuccess || (e = launch_gemv(h->lc, gemv_fmt(h), gu)) != cudaSuccess) return e;

        GemvArgs dn{};
        dn.mode = 1; dn.w = L.wd; dn.s = L.sd; dn.N = c.hidden; dn.K = c.mlp; dn.x = h->u; dn.y = h->x;
        dn.stats_in = st_gu; dn.stats_out = st_down;
        if (ofold) {
            dn.fold = h->o_d;
            dn.fold_add = 1;
        }
        dn.stats_gamma = (const uint16_t *)(l + 1 < c.n_layers ? h->layers[l + 1].attn_norm : h->w.final_norm);
        dn.tl = slot(LLM_KIND_DOWN);
        if ((h->l2pf & kL2pfDownNext) && l + 1 < c.n_layers) {  // the next layer's QKV and o_proj codes
            const llm_layer_weights &Nx = h->layers[l + 1];
            dn.pf[0] = {Nx.wq, code_bytes(h, rq, c.hidden)};
            dn.pf[1] = {Nx.wk, code_bytes(h, rkv, c.hidden)};
            dn.pf[2] = {Nx.wv, code_bytes(h, rkv, c.hidden)};
            dn.pf[3] = {Nx.wo, code_bytes(h, c.hidden, rq)};
        }
        if ((e = mark()) != cudaSuccess || (e = launch_gemv(h->lc, gemv_fmt(h), dn)) != cudaSuccess) return e;
    }
    LmHeadArgs la{};
    const bool int8_head = h->fmt == kFmtInt8 && !c.tied_lm_head;
    la.fmt = int8_head ? kFmtInt8 : kFmtBf16;
    la.w = c.tied_lm_head ? h->w.embed : h->w.lm_head;
    la.scale = int8_head ? (const float *)h->w.lm_scale : nullptr;
    la.gamma = (const uint16_t *)h->w.final_norm;
    la.eps = c.rms_eps; la.N = c.vocab; la.K = c.hidden; la.x = h->x; la.logits = h->logits;
    la.part_val = h->lm_part_val; la.part_idx = h->lm_part_idx; la.counter = h->lm_counter;
    la.token_out = &h->st->last_token; la.st = h->st; la.advance = 1;
    la.stats_in = fmlp ? nullptr : st_down;
    la.x2 = fmlp ? h->mlp_d : nullptr;
    if (h->sampling) {  // the sampler takes the token and advances the state
        la.token_out = h->samp_scratch; la.st = nullptr; la.advance = 0;
    }
    la.tl = slot(LLM_KIND_LM_HEAD);
    if ((e = mark()) != cudaSuccess || (e = launch_lm_head(h->lc, la, h->lm_grid)) != cudaSuccess) return e;
    if (h->sampling) {
        SampleArgs sa = sampler_args(h);
        sa.tl = slot(LLM_KIND_SAMPLER);
        if ((e = launch_sample(h->lc, sa)) != cudaSuccess) return e;
    }
    if (n_launch) *n_launch = kl;
    return mark();
}

// (Re)capture the whole step into the graph with the current launch settings.
int capture(llm_t *h) {
    if (h->exec) cudaGraphExecDestroy(h->exec);
    if (h->graph) cudaGraphDestroy(h->graph);
    h->exec = nullptr;
    h->graph = nullptr;
    if (cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return LLM_ERR_CUDA;
    cudaError_t ce = enqueue_step(h);
    cudaError_t ee = cudaStreamEndCapture(h->stream, &h->graph);
    if (ce != cudaSuccess || ee != cudaSuccess) return LLM_ERR_CUDA;
    if (cudaGraphInstantiate(&h->exec, h->graph, 0) != cudaSuccess) return LLM_ERR_CUDA;
    return LLM_OK;
}

int run_step(llm_t *h) {
    cudaError_t e = h->use_graph ? cudaGraphLaunch(h->exec, h->stream) : enqueue_step(h);
    return e == cudaSuccess ? LLM_OK : LLM_ERR_CUDA;
}

// Fill the persistent kernel's parameters; leaves h->step_ok false (kernel
// chain) when the shapes are outside what it supports.
int plan_step(llm_t *h, int n_sm) {
    const llm_config &c = h->cfg;
    StepParams &p = h->sp;
    p = StepParams{};
    p.L = c.n_layers;
    p.h = c.hidden;
    p.Hq = c.n_q_heads;
    p.Hkv = c.n_kv_heads;
    p.d = c.head_dim;
    p.F = c.mlp;
    p.V = c.vocab;
    p.eps = c.rms_eps;
    p.embed = (const uint16_t *)h->w.embed;
    p.final_norm = (const uint16_t *)h->w.final_norm;
    const bool int8_head = h->fmt == kFmtInt8 && !c.tied_lm_head;
    p.lm_w = c.tied_lm_head ? h->w.embed : h->w.lm_head;
    p.lm_scale = int8_head ? (const float *)h->w.lm_scale : nullptr;
    p.page_table = h->page_table;
    p.n_pages = h->n_pages;
    p.rope_cs = h->rope_cs;
    p.k_pool = h->k_pool;
    p.v_pool = h->v_pool;
    p.st = h->st;
    p.x = h->x;
    p.raw = h->raw;
    p.q = h->q;
    p.attn = h->attn;
    p.u = h->u;
    p.logits = h->logits;
    p.part_o = h->part_o;
    p.part_ml = h->part_ml;
    p.lm_val = h->lm_part_val;
    p.lm_idx = h->lm_part_idx;
    p.wait_ns = 1000000000ull;  // 1 s: a step takes about a millisecond
    p.counter_wait_ns = p.wait_ns;
    p.test_extra_arrivals = 0;
    p.inflight = kStepMaxSlots; // ring items in flight: enough bytes to cover the HBM latency
    int max_smem = 0;
    if (cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, h->device) != cudaSuccess)
        return LLM_ERR_CUDA;
    h->step_ok = step_plan(p, h->fmt, int8_head ? kFmtInt8 : kFmtBf16, n_sm, max_smem, h->sl);
    if (!h->step_ok) return LLM_OK;
    int per_sm = 0;
    if (step_occupancy(h->sl, &per_sm) != cudaSuccess || per_sm < 1) {
        cudaGetLastError();
        h->step_ok = false;
        return LLM_OK;
    }
    std::vector<StepLayer> ly(c.n_layers);
    std::vector<CUtensorMap> maps((size_t)c.n_layers * kMapCount);
    if (dalloc(&h->d_maps, maps.size()) != cudaSuccess) return LLM_ERR_CUDA;
    const int rq = c.n_q_heads * c.head_dim, rkv = c.n_kv_heads * c.head_dim;
    for (int l = 0; l < c.n_layers; ++l) {
        const llm_layer_weights &L = h->layers[l];
        StepLayer &S = ly[l];
        CUtensorMap *m = maps.data() + (size_t)l * kMapCount;
        if (step_encode_weight_map(m + kMapQ, L.wq, rq, p.geo[kPhQkv], kStepLines) != cudaSuccess ||
            step_encode_weight_map(m + kMapK, L.wk, rkv, p.geo[kPhQkv], kStepLines) != cudaSuccess ||
            step_encode_weight_map(m + kMapV, L.wv, rkv, p.geo[kPhQkv], kStepLines) != cudaSuccess ||
            step_encode_weight_map(m + kMapO, L.wo, c.hidden, p.geo[kPhO], kStepLines) != cudaSuccess ||
            step_encode_weight_map(m + kMapGate, L.wg, c.mlp, p.geo[kPhGu], kStepLines / 2) != cudaSuccess ||
            step_encode_weight_map(m + kMapUp, L.wu, c.mlp, p.geo[kPhGu], kStepLines / 2) != cudaSuccess ||
            step_encode_weight_map(m + kMapDown, L.wd, c.hidden, p.geo[kPhDown], kStepLines) != cudaSuccess) {
            h->step_ok = false;
            return LLM_OK;
        }
        S.tm = h->d_maps + (size_t)l * kMapCount;
        S.w[0] = L.wq; S.w[1] = L.wk; S.w[2] = L.wv;
        S.s[0] = L.sq; S.s[1] = L.sk; S.s[2] = L.sv;
        if (c.qkv_bias) {
            S.b[0] = (const uint16_t *)L.bq;
            S.b[1] = (const uint16_t *)L.bk;
            S.b[2] = (const uint16_t *)L.bv;
        }
        S.wo = L.wo; S.so = L.so; S.wg = L.wg; S.sg = L.sg; S.wu = L.wu; S.su = L.su; S.wd = L.wd; S.sd = L.sd;
        S.attn_norm = (const uint16_t *)L.attn_norm;
        S.mlp_norm = (const uint16_t *)L.mlp_norm;
        if (c.qk_norm) {
            S.q_norm = (const uint16_t *)L.q_norm;
            S.k_norm = (const uint16_t *)L.k_norm;
        }
    }
    const size_t n_sync = (size_t)c.n_layers * kSyncStride + 1;
    const size_t kv_rows = (size_t)c.n_layers * h->n_pages * c.n_kv_heads * kPageTokens;
    if (dalloc(&h->d_layers, ly.size()) != cudaSuccess || dalloc(&h->step_sync, n_sync) != cudaSuccess ||
        dalloc(&h->prof, (size_t)5 * c.n_layers + 2) != cudaSuccess ||
        cudaMemcpyAsync(h->d_layers, ly.data(), ly.size() * sizeof(StepLayer), cudaMemcpyHostToDevice,
                        h->stream) != cudaSuccess ||
        cudaMemcpyAsync(h->d_maps, maps.data(), maps.size() * sizeof(CUtensorMap), cudaMemcpyHostToDevice,
                        h->stream) != cudaSuccess ||
        cudaMemsetAsync(h->step_sync, 0, n_sync * sizeof(int), h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    p.layers = h->d_layers;
    p.sync = h->step_sync;
    if (step_encode_kv_maps(p, kv_rows) != cudaSuccess ||
        step_encode_weight_map(&p.tm_lm, p.lm_w, c.vocab, p.geo[kPhLm], kStepLines) != cudaSuccess) {
        h->step_ok = false;
        return LLM_OK;
    }
    h->persistent = false;  // opt-in (llm_set_persistent) until it outpaces the kernel chain
    return LLM_OK;
}

int fetch_token(llm_t *h, int32_t *out) {
    if (cudaMemcpyAsync(h->pinned + 2, &h->st->last_token, 2 * sizeof(int32_t),
                        cudaMemcpyDeviceToHost, h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    if (h->pinned[3] != kErrNone) return h->pinned[3] == kErrTimeout ? LLM_ERR_TIMEOUT : LLM_ERR_DEVICE;
    if (out) *out = h->pinned[2];
    return LLM_OK;
}

// ---- batched prefill -------------------------------------------------------------
// Rows of a prompt chunk go through the layers as GEMMs: RMSNorm -> fp16 rows,
// tcgen05 GEMMs that dequantize each weight code tile in shared memory, with a
// fused epilogue (QKV store, o_proj/down residual add, gate/up SiLU * mul),
// causal flash attention over the paged cache.  The last row of the prompt
// then runs the decode step's LM head (+ argmax), which also advances the
// device state.
constexpr int kPrefillChunk = 1024;

bool prefill_shapes_ok(const llm_config &c) {
    const int d = c.head_dim, rq = c.n_q_heads * d, nq = (c.n_q_heads + 2 * c.n_kv_heads) * d;
    const int rkv = c.n_kv_heads * d;
    // every 128-row weight tile lies in one matrix (q, k, v stacked); K % 128 for the code tiles
    return rq % kTcBN == 0 && rkv % kTcBN == 0 && nq % kTcBN == 0 && c.hidden % kTcBN == 0 && c.mlp % 64 == 0 &&
           c.hidden % 128 == 0 && rq % 128 == 0 && c.mlp % 128 == 0;
}

int prefill_alloc(llm_t *h) {
    if (h->pf_ready) return LLM_OK;
    const llm_config &c = h->cfg;
    const int d = c.head_dim, rq = c.n_q_heads * d, nq = (c.n_q_heads + 2 * c.n_kv_heads) * d;
    const int R = ((c.max_context < kPrefillChunk ? c.max_context : kPrefillChunk) + kTcBM - 1) / kTcBM * kTcBM;
    h->pf_rows = R;
    const size_t arow = (size_t)std::max(c.hidden, rq);
    bool ok = dalloc(&h->pf_x, (size_t)R * c.hidden) == cudaSuccess &&
              dalloc(&h->pf_raw, (size_t)R * nq) == cudaSuccess && dalloc(&h->pf_a, (size_t)R * arow) == cudaSuccess &&
              dalloc(&h->pf_u, (size_t)R * c.mlp) == cudaSuccess && dalloc(&h->pf_qh, (size_t)R * rq) == cudaSuccess &&
              dalloc(&h->pf_ql, (size_t)R * rq) == cudaSuccess && dalloc(&h->pf_tok, (size_t)R) == cudaSuccess;
    if (!ok) return LLM_ERR_CUDA;
    // rows past a chunk's end are read by the GEMMs (their outputs are dropped): keep them finite
    ok = cudaMemsetAsync(h->pf_a, 0, (size_t)R * arow * 2, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->pf_u, 0, (size_t)R * c.mlp * 2, h->stream) == cudaSuccess &&
         tc_act_map(&h->pf_map_ah, h->pf_a, R, c.hidden) == cudaSuccess &&
         tc_act_map(&h->pf_map_aq, h->pf_a, R, rq) == cudaSuccess &&
         tc_act_map(&h->pf_map_u, h->pf_u, R, c.mlp) == cudaSuccess;
    if (!ok) return LLM_ERR_CUDA;
    // code-tile maps of every weight matrix (the GEMMs dequantize in shared memory)
    const int rkv = c.n_kv_heads * d;
    h->pf_wmaps.assign((size_t)c.n_layers * 7, CUtensorMap{});
    for (int l = 0; l < c.n_layers; ++l) {
        const llm_layer_weights &L = h->layers[l];
        CUtensorMap *m = h->pf_wmaps.data() + (size_t)l * 7;
        ok = tc_weight_map(m + 0, L.wq, h->fmt, rq, c.hidden, kTcBN) == cudaSuccess &&
             tc_weight_map(m + 1, L.wk, h->fmt, rkv, c.hidden, kTcBN) == cudaSuccess &&
             tc_weight_map(m + 2, L.wv, h->fmt, rkv, c.hidden, kTcBN) == cudaSuccess &&
             tc_weight_map(m + 3, L.wo, h->fmt, c.hidden, rq, kTcBN) == cudaSuccess &&
             tc_weight_map(m + 4, L.wg, h->fmt, c.mlp, c.hidden, kTcBN / 2) == cudaSuccess &&
             tc_weight_map(m + 5, L.wu, h->fmt, c.mlp, c.hidden, kTcBN / 2) == cudaSuccess &&
             tc_weight_map(m + 6, L.wd, h->fmt, c.hidden, c.mlp, kTcBN) == cudaSuccess;
        if (!ok) return LLM_ERR_CUDA;
    }
    h->pf_ready = true;
    return LLM_OK;
}

// One chunk of m prompt rows at positions pos0 .. pos0 + m - 1 (tokens already
// on the device in pf_tok).  Leaves the residual rows in pf_x.
cudaError_t prefill_chunk(llm_t *h, int m, int pos0) {
    const llm_config &c = h->cfg;
    const int d = c.head_dim, rq = c.n_q_heads * d, rkv = c.n_kv_heads * d, nq = rq + 2 * rkv;
    cudaStream_t st = h->stream;
    int *err = &h->st->err;
    cudaError_t e;
    // A (fp16 rows) x the weight codes of up to three stacked matrices, or an interleaved pair
    auto gemm = [&](const CUtensorMap &am, const CUtensorMap *w0, const CUtensorMap *w1, const CUtensorMap *w2,
                    TcQuantB qb, int N, int K, int mode, float *cc, int ldc, uint16_t *hh, int ldh) {
        const CUtensorMap wm[3] = {*w0, w1 ? *w1 : *w0, w2 ? *w2 : *w0};
        qb.fmt = h->fmt;
        TcGemmArgs g{};
        g.M = m; g.N = N; g.K = K; g.mode = mode; g.c = cc; g.ldc = ldc; g.h = hh; g.ldh = ldh;
        g.err = err; g.wait_ns = 1000000000ull;
        return launch_tc_gemm_q(st, am, wm, qb, g, true);
    };
    auto one = [](const void *scale, int rows) {
        TcQuantB q{};
        q.n_seg = 1; q.seg_rows[0] = rows; q.scale[0] = scale;
        return q;
    };
    if ((e = launch_embed_rows(st, (const uint16_t *)h->w.embed, h->pf_tok, m, c.hidden, h->pf_x)) != cudaSuccess)
        return e;
    for (int l = 0; l < c.n_layers; ++l) {
        const llm_layer_weights &L = h->layers[l];
        uint16_t *kp = h->k_pool + (size_t)l * h->layer_kv_elems, *vp = h->v_pool + (size_t)l * h->layer_kv_elems;
        const CUtensorMap *wm = h->pf_wmaps.data() + (size_t)l * 7;
        TcQuantB qkv{};
        qkv.n_seg = 3;
        qkv.seg_rows[0] = rq; qkv.seg_rows[1] = rkv; qkv.seg_rows[2] = rkv;
        qkv.scale[0] = L.sq; qkv.scale[1] = L.sk; qkv.scale[2] = L.sv;
        TcQuantB gu{};
        gu.interleave = 1;
        gu.seg_rows[0] = gu.seg_rows[1] = c.mlp;
        gu.scale[0] = L.sg; gu.scale[1] = L.su;
        if ((e = launch_rmsnorm_rows(st, h->pf_x, (const uint16_t *)L.attn_norm, c.rms_eps, m, c.hidden, h->pf_a)) ||
            (e = gemm(h->pf_map_ah, wm + 0, wm + 1, wm + 2, qkv, nq, c.hidden, kEpiStore, h->pf_raw, nq, nullptr, 0)))
            return e;
        QkvRowsArgs qa{};
        qa.raw = h->pf_raw;
        if (c.qkv_bias) {
            qa.bq = (const uint16_t *)L.bq;
            qa.bk = (const uint16_t *)L.bk;
            qa.bv = (const uint16_t *)L.bv;
        }
        if (c.qk_norm) {
            qa.q_gain = (const uint16_t *)L.q_norm;
            qa.k_gain = (const uint16_t *)L.k_norm;
        }
        qa.eps = c.rms_eps; qa.n = m; qa.pos0 = pos0; qa.Hq = c.n_q_heads; qa.Hkv = c.n_kv_heads; qa.d = d;
        qa.rope_cs = h->rope_cs; qa.k_pool = kp; qa.v_pool = vp; qa.page_table = h->page_table;
        qa.n_pages = h->n_pages; qa.q_hi = h->pf_qh; qa.q_lo = h->pf_ql; qa.err = err;
        AttnRowsArgs aa{};
        aa.q_hi = h->pf_qh; aa.q_lo = h->pf_ql; aa.k_pool = kp; aa.v_pool = vp; aa.page_table = h->page_table;
        aa.n_pages = h->n_pages; aa.n = m; aa.pos0 = pos0; aa.Hq = c.n_q_heads; aa.Hkv = c.n_kv_heads; aa.d = d;
        aa.out = h->pf_a; aa.err = err;
        if ((e = launch_qkv_rows(st, qa)) || (e = launch_attn_rows(st, aa)) ||
            (e = gemm(h->pf_map_aq, wm + 3, nullptr, nullptr, one(L.so, c.hidden), c.hidden, rq, kEpiAdd, h->pf_x,
                      c.hidden, nullptr, 0)) ||
            (e = launch_rmsnorm_rows(st, h->pf_x, (const uint16_t *)L.mlp_norm, c.rms_eps, m, c.hidden, h->pf_a)) ||
            (e = gemm(h->pf_map_ah, wm + 4, wm + 5, nullptr, gu, 2 * c.mlp, c.hidden, kEpiSwiGlu, nullptr, 0,
                      h->pf_u, c.mlp)) ||
            (e = gemm(h->pf_map_u, wm + 6, nullptr, nullptr, one(L.sd, c.hidden), c.hidden, c.mlp, kEpiAdd, h->pf_x,
                      c.hidden, nullptr, 0)))
            return e;
    }
    return cudaSuccess;
}

int prefill_batched(llm_t *h, const int32_t *tokens, int n, int32_t *first_token) {
    int rc = prefill_alloc(h);
    if (rc != LLM_OK) return rc;
    const llm_config &c = h->cfg;
    int last_rows = 0;
    for (int off = 0; off < n; off += h->pf_rows) {
        const int m = n - off < h->pf_rows ? n - off : h->pf_rows;
        if (cudaMemcpyAsync(h->pf_tok, tokens + off, (size_t)m * sizeof(int32_t), cudaMemcpyHostToDevice,
                            h->stream) != cudaSuccess ||
            prefill_chunk(h, m, h->seq_len + off) != cudaSuccess)
            return LLM_ERR_CUDA;
        last_rows = m;
    }
    // the last prompt row -> final RMSNorm -> LM head + argmax; the state moves to seq_len + n
    k_set_state<<<1, 1, 0, h->stream>>>(h->st, -1, h->seq_len + n - 1, 0);
    if (cudaGetLastError() != cudaSuccess ||
        cudaMemcpyAsync(h->x, h->pf_x + (size_t)(last_rows - 1) * c.hidden, (size_t)c.hidden * sizeof(float),
                        cudaMemcpyDeviceToDevice, h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    LmHeadArgs la{};
    const bool int8_head = h->fmt == kFmtInt8 && !c.tied_lm_head;
    la.fmt = int8_head ? kFmtInt8 : kFmtBf16;
    la.w = c.tied_lm_head ? h->w.embed : h->w.lm_head;
    la.scale = int8_head ? (const float *)h->w.lm_scale : nullptr;
    la.gamma = (const uint16_t *)h->w.final_norm;
    la.eps = c.rms_eps; la.N = c.vocab; la.K = c.hidden; la.x = h->x; la.logits = h->logits;
    la.part_val = h->lm_part_val; la.part_idx = h->lm_part_idx; la.counter = h->lm_counter;
    la.token_out = &h->st->last_token; la.st = h->st; la.advance = 1;
    if (h->sampling) {
        la.token_out = h->samp_scratch; la.st = nullptr; la.advance = 0;
    }
    LaunchCfg lc = h->lc;
    lc.pdl = false;
    if (launch_lm_head(lc, la, h->lm_grid) != cudaSuccess) return LLM_ERR_CUDA;
    if (h->sampling && launch_sample(lc, sampler_args(h)) != cudaSuccess) return LLM_ERR_CUDA;
    return fetch_token(h, first_token);
}

}  // namespace

namespace qd {
// llm_create_from_file hands the handle the weights' device copy (freed by llm_destroy).
void adopt_weight_buffer(llm_t *h, void *dev) { h->weight_buffer = dev; }
}  // namespace qd

extern "C" {

#ifndef QD_BUILD_ID
#define QD_BUILD_ID "unknown"
#endif
const char *llm_build_id(void) { return QD_BUILD_ID; }

const char *llm_status_str(int s) {
    switch (s) {
        case LLM_OK: return "ok";
        case LLM_ERR_ARG: return "invalid argument";
        case LLM_ERR_LAYOUT: return "packed layout does not match the weight format";
        case LLM_ERR_CONTEXT_FULL: return "context full";
        case LLM_ERR_CUDA: return "CUDA runtime error";
        case LLM_ERR_TIMEOUT: return "device wait timed out";
        case LLM_ERR_DEVICE: return "device-side check failed";
        case LLM_ERR_STATE: return "call out of order";
        case LLM_ERR_FORMAT: return "not a model file, or a corrupt or truncated one";
        case LLM_ERR_IO: return "file could not be opened, read or written";
        default: return "unknown status";
    }
}

int llm_create(const llm_config *cfg, const llm_weights *weights, void *cuda_stream, llm_t **out) {
    if (!out) return LLM_ERR_ARG;
    *out = nullptr;
    int rc = validate(cfg, weights);
    if (rc != LLM_OK) return rc;
    llm_t *h = new (std::nothrow) llm_t();
    if (!h) return LLM_ERR_CUDA;
    h->cfg = *cfg;
    h->fmt = cfg->weight_format == LLM_FMT_INT4_G128 ? kFmtInt4 : kFmtInt8;
    h->layers.assign(weights->layers, weights->layers + cfg->n_layers);
    h->w = *weights;
    h->w.layers = nullptr;

    auto fail = [&](int code) {
        free_all(h);
        delete h;
        return code;
    };
    if (cudaGetDevice(&h->device) != cudaSuccess) return fail(LLM_ERR_CUDA);
    int n_sm = 0;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess)
        return fail(LLM_ERR_CUDA);
    if (cuda_stream) {
        h->stream = (cudaStream_t)cuda_stream;
    } else {
        if (cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking) != cudaSuccess)
            return fail(LLM_ERR_CUDA);
        h->own_stream = true;
    }
    h->lc.stream = h->stream;
    h->lc.pdl = true;   // measured: early dependent launch saves 0.05-0.1 ms per 7B step
    h->lc.n_sm = n_sm;

    const llm_config &c = h->cfg;
    const int d = c.head_dim, G = c.n_q_heads / c.n_kv_heads;
    h->n_pages = (c.max_context + kPageTokens - 1) / kPageTokens;
    h->layer_kv_elems = (size_t)h->n_pages * c.n_kv_heads * kPageTokens * d;
    const AttnPlan ap = plan_attention(n_sm, c.n_q_heads, c.n_kv_heads, d, h->n_pages);
    h->P = ap.P;
    h->attn_cs = ap.cs;
    h->fused_ok = qkv_attn_fusable(h->fmt, c.n_q_heads, c.n_kv_heads, d, c.hidden, c.qk_norm != 0, ap);
    h->fused = false;  // measured slower than the separate kernels at 7B (1.83 vs 1.69 ms/token)
    h->o_fold_ok = attn_fold_ok(h->fmt, c.n_q_heads, c.n_kv_heads, d, c.hidden, ap);
    h->lm_grid = lm_head_grid(h->lc, c.vocab);
    const int P_alloc = h->P > n_sm / c.n_kv_heads ? h->P : n_sm / c.n_kv_heads + 1;
    const int lm_alloc = h->lm_grid > n_sm ? h->lm_grid : n_sm;
    const size_t kv_elems = h->layer_kv_elems * c.n_layers;
    const int rows_qkv = (c.n_q_heads + 2 * c.n_kv_heads) * d;
    const int heads_qkv = c.n_q_heads + 2 * c.n_kv_heads;
    bool ok = dalloc(&h->k_pool, kv_elems) == cudaSuccess && dalloc(&h->v_pool, kv_elems) == cudaSuccess &&
              dalloc(&h->page_table, h->n_pages) == cudaSuccess &&
              dalloc(&h->rope_cs, (size_t)c.max_context * (d / 2)) == cudaSuccess &&
              dalloc(&h->st, 1) == cudaSuccess && dalloc(&h->x, c.hidden) == cudaSuccess &&
              dalloc(&h->raw, rows_qkv) == cudaSuccess && dalloc(&h->q, c.n_q_heads * d) == cudaSuccess &&
              dalloc(&h->attn, c.n_q_heads * d) == cudaSuccess && dalloc(&h->u, c.mlp) == cudaSuccess &&
              dalloc(&h->logits, c.vocab) == cudaSuccess && dalloc(&h->head_cnt, heads_qkv) == cudaSuccess &&
              dalloc(&h->attn_cnt, c.n_kv_heads) == cudaSuccess && dalloc(&h->lm_counter, 1) == cudaSuccess &&
              dalloc(&h->lm_part_idx, lm_alloc) == cudaSuccess &&
              dalloc(&h->lm_part_val, lm_alloc) == cudaSuccess &&
              dalloc(&h->part_o, (size_t)c.n_kv_heads * P_alloc * G * d) == cudaSuccess &&
              dalloc(&h->part_ml, (size_t)c.n_kv_heads * P_alloc * G * 2) == cudaSuccess &&
              dalloc(&h->stats, (size_t)8 * kStatSlots) == cudaSuccess &&
              dalloc(&h->kv_new, (size_t)2 * c.n_kv_heads * d) == cudaSuccess &&
              dalloc(&h->samp_scratch, 1) == cudaSuccess &&
              cudaMallocHost(reinterpret_cast<void **>(&h->pinned), 8 * sizeof(int32_t)) == cudaSuccess;
    if (!ok) return fail(LLM_ERR_CUDA);

    // Zeroed pools (slots past the sequence never hold NaN), counters at zero.
    ok = cudaMemsetAsync(h->k_pool, 0, kv_elems * 2, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->v_pool, 0, kv_elems * 2, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->st, 0, sizeof(DevState), h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->head_cnt, 0, heads_qkv * sizeof(int), h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->attn_cnt, 0, c.n_kv_heads * sizeof(int), h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->lm_counter, 0, sizeof(int), h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->logits, 0, c.vocab * sizeof(float), h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->stats, 0, (size_t)8 * kStatSlots * sizeof(float), h->stream) == cudaSuccess;
    if (!ok) return fail(LLM_ERR_CUDA);

    // Identity page table and the RoPE table: angle pos * base^(-2i/d) formed in double.
    std::vector<int32_t> pt(h->n_pages);
    for (int i = 0; i < h->n_pages; ++i) pt[i] = i;
    std::vector<float2> cs((size_t)c.max_context * (d / 2));
    for (int p = 0; p < c.max_context; ++p)
        for (int i = 0; i < d / 2; ++i) {
            const double theta = std::pow((double)c.rope_base, -2.0 * (double)i / (double)d);
            const double ang = (double)p * theta;
            cs[(size_t)p * (d / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    ok = cudaMemcpyAsync(h->page_table, pt.data(), pt.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                         h->stream) == cudaSuccess &&
         cudaMemcpyAsync(h->rope_cs, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice,
                         h->stream) == cudaSuccess &&
         cudaStreamSynchronize(h->stream) == cudaSuccess;
    if (!ok) return fail(LLM_ERR_CUDA);

    // The MLP block as one kernel: W_down of every layer repacked unit-major (the
    // layout k_mlp streams), D zeroed.
    h->mlp_ok = mlp_shape_ok(h->fmt, c.hidden, c.mlp);
    if (h->mlp_ok) {
        h->mlp_w_bytes = (h->fmt == kFmtInt4 ? (size_t)c.hidden * c.mlp / 2 : (size_t)c.hidden * c.mlp);
        h->mlp_s_bytes = h->fmt == kFmtInt4 ? (((size_t)c.hidden * (c.mlp / kGroup) * 2 + 255) & ~(size_t)255) : 0;
        const size_t per = h->mlp_w_bytes + h->mlp_s_bytes;
        ok = cudaMalloc((void **)&h->mlp_buf, per * c.n_layers) == cudaSuccess &&
             dalloc(&h->mlp_d, c.hidden) == cudaSuccess &&
             cudaMemsetAsync(h->mlp_d, 0, (size_t)c.hidden * sizeof(long long), h->stream) == cudaSuccess;
        for (int l = 0; ok && l < c.n_layers; ++l) {
            char *dst = h->mlp_buf + (size_t)l * per;
            ok = mlp_repack_down(h->fmt, h->layers[l].wd, h->layers[l].sd, c.hidden, c.mlp, dst,
                                 h->fmt == kFmtInt4 ? dst + h->mlp_w_bytes : nullptr, h->stream) == cudaSuccess;
        }
        if (!ok || cudaStreamSynchronize(h->stream) != cudaSuccess) return fail(LLM_ERR_CUDA);
        // Default where it measured faster than the two GEMV kernels: narrow models,
        // whose down GEMV has few row tiles per SM (1.5B shape: 1.018 vs 1.069 ms per
        // token); on the 7B shape the in-CTA down phase is slower than the separate
        // kernel (2.07 vs 1.75 ms per token).
        h->mlp_fused = c.hidden <= 2048;
    }

    // o_proj folded into the attention: its pending output, zero between steps
    if (h->o_fold_ok) {
        std::vector<AttnFold> fa((size_t)c.n_layers);
        const AttnPlan ap{h->P, h->attn_cs};
        if (dalloc(&h->o_d, c.hidden) != cudaSuccess ||
            cudaMemsetAsync(h->o_d, 0, (size_t)c.hidden * sizeof(long long), h->stream) != cudaSuccess ||
            cudaMalloc((void **)&h->o_fold_args, fa.size() * sizeof(AttnFold)) != cudaSuccess)
            return fail(LLM_ERR_CUDA);
        for (int l = 0; l < c.n_layers; ++l)
            if (attn_fold_args(fa[l], h->layers[l].wo, (const uint16_t *)h->layers[l].so, h->o_d, c.n_q_heads,
                               c.n_kv_heads, d, c.hidden, ap) != cudaSuccess)
                return fail(LLM_ERR_CUDA);
        if (cudaMemcpyAsync(h->o_fold_args, fa.data(), fa.size() * sizeof(AttnFold), cudaMemcpyHostToDevice,
                            h->stream) != cudaSuccess ||
            cudaStreamSynchronize(h->stream) != cudaSuccess)
            return fail(LLM_ERR_CUDA);
        h->o_fold = false;
    }

    if (plan_step(h, n_sm) != LLM_OK) return fail(LLM_ERR_CUDA);
    h->pf_ok = prefill_shapes_ok(c);

    // Capture the whole step once (the kernel chain if the persistent kernel
    // cannot be captured here).
    if (capture(h) != LLM_OK) {
        cudaGetLastError();
        if (!h->persistent) return fail(LLM_ERR_CUDA);
        h->persistent = false;
        h->step_ok = false;
        if (capture(h) != LLM_OK) return fail(LLM_ERR_CUDA);
    }
    *out = h;
    return LLM_OK;
}

void llm_destroy(llm_t *h) {
    if (!h) return;
    cudaStreamSynchronize(h->stream);
    free_all(h);
    if (h->weight_buffer) cudaFree(h->weight_buffer);
    delete h;
}

int llm_set_graph_mode(llm_t *h, int32_t use_graph) {
    if (!h) return LLM_ERR_ARG;
    h->use_graph = use_graph != 0;
    return LLM_OK;
}

int llm_set_persistent(llm_t *h, int32_t on) {
    if (!h) return LLM_ERR_ARG;
    if (on && (!h->step_ok || h->sampling || h->act_int8)) return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->persistent = on != 0;
    return capture(h);
}

int llm_set_o_fold(llm_t *h, int32_t on) {
    if (!h || (on && !h->o_fold_ok)) return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->o_fold = on != 0;
    // o_d is zero between completed steps either way: each layer's down zeroes it
    return capture(h);
}

int llm_get_o_fold(llm_t *h, int32_t *on) {
    if (!h || !on) return LLM_ERR_ARG;
    *on = h->o_fold ? 1 : 0;
    return LLM_OK;
}

int llm_set_fused_mlp(llm_t *h, int32_t on) {
    if (!h || (on && !h->mlp_ok)) return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->mlp_fused = on != 0;
    // D may hold a finished step's last-layer output: the next step's first o_proj
    // zeroes it either way, and the unfused chain never reads it.
    return capture(h);
}

int llm_step_kinds(llm_t *h, int32_t *kinds, int32_t cap, int32_t *n) {
    if (!h || !kinds || !n) return LLM_ERR_ARG;
    *n = (int32_t)h->kinds.size();
    if (h->persistent) {
        *n = 0;
        return LLM_OK;
    }
    if (cap < *n) return LLM_ERR_ARG;
    for (int i = 0; i < *n; ++i) kinds[i] = h->kinds[i];
    return LLM_OK;
}

int llm_set_l2_prefetch(llm_t *h, int32_t flags) {
    if (!h || flags < 0 || flags > kL2pfAll) return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->l2pf = flags;
    return capture(h);
}

int llm_debug_step_wait(llm_t *h, int32_t extra_arrivals, int64_t counter_wait_ns) {
    if (!h || !h->step_ok || extra_arrivals < 0 || extra_arrivals > 1 || counter_wait_ns < 1000 ||
        counter_wait_ns > 1000000000ll)
        return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->sp.test_extra_arrivals = extra_arrivals;
    h->sp.counter_wait_ns = (unsigned long long)counter_wait_ns;
    return h->persistent ? capture(h) : LLM_OK;
}

int llm_set_act_int8(llm_t *h, int32_t on) {
    if (!h) return LLM_ERR_ARG;
    if (on && (h->fmt != kFmtInt4 || h->persistent)) return LLM_ERR_ARG;
    if (on && (!gemv_shape_ok(kFmtInt4A8, h->cfg.hidden, h->cfg.n_q_heads * h->cfg.head_dim, 1) ||
               !gemv_shape_ok(kFmtInt4A8, h->cfg.mlp, h->cfg.hidden, 2) ||
               !gemv_shape_ok(kFmtInt4A8, h->cfg.hidden, h->cfg.mlp, 1)))
        return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->act_int8 = on != 0;
    return capture(h);
}

int llm_set_sampling(llm_t *h, float temperature, int32_t top_k, float top_p, uint64_t seed) {
    if (!h) return LLM_ERR_ARG;
    const bool on = temperature > 0.f;
    if (on && (h->persistent || top_k < 1 || top_k > kMaxTopK || top_k > h->cfg.vocab || !(top_p > 0.f) ||
               top_p > 1.f || !(temperature < INFINITY)))
        return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->sampling = on;
    h->samp_t = temperature; h->samp_k = top_k; h->samp_p = top_p; h->samp_seed = seed;
    return capture(h);
}

int llm_set_prefill_batched(llm_t *h, int32_t on) {
    if (!h) return LLM_ERR_ARG;
    if (on && !h->pf_ok) return LLM_ERR_ARG;
    h->pf_batched = on != 0;
    return LLM_OK;
}

int llm_set_fused_attention(llm_t *h, int32_t on) {
    if (!h || (on && !h->fused_ok)) return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->fused = on != 0;
    return capture(h);
}

int llm_set_pdl(llm_t *h, int32_t use_pdl) {
    if (!h) return LLM_ERR_ARG;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->lc.pdl = use_pdl != 0;
    return capture(h);
}

int llm_prefill(llm_t *h, const int32_t *tokens, int32_t n, int32_t *first_token) {
    if (!h || !tokens || n <= 0) return LLM_ERR_ARG;
    for (int i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab) return LLM_ERR_ARG;
    if ((int64_t)h->seq_len + n > h->cfg.max_context) return LLM_ERR_CONTEXT_FULL;
    if (h->pf_ok && h->pf_batched && n >= 2) {
        int rc = prefill_batched(h, tokens, n, first_token);
        if (rc != LLM_OK) return rc;
        h->seq_len += n;
        h->have_token = true;
        h->stepped = true;
        return LLM_OK;
    }
    for (int i = 0; i < n; ++i) {
        k_set_state<<<1, 1, 0, h->stream>>>(h->st, tokens[i], i == 0 ? h->seq_len : -1, 0);
        if (cudaGetLastError() != cudaSuccess) return LLM_ERR_CUDA;
        int rc = run_step(h);
        if (rc != LLM_OK) return rc;
    }
    int rc = fetch_token(h, first_token);
    if (rc != LLM_OK) return rc;
    h->seq_len += n;
    h->have_token = true;
    h->stepped = true;
    return LLM_OK;
}

int llm_decode_step(llm_t *h, int32_t forced_input, int32_t *out_token) {
    if (!h) return LLM_ERR_ARG;
    if (forced_input >= h->cfg.vocab) return LLM_ERR_ARG;
    if (h->seq_len >= h->cfg.max_context) return LLM_ERR_CONTEXT_FULL;
    if (forced_input < 0 && !h->have_token) return LLM_ERR_STATE;
    if (forced_input >= 0) {
        h->pinned[0] = forced_input;
        if (cudaMemcpyAsync(&h->st->token, h->pinned, sizeof(int32_t), cudaMemcpyHostToDevice,
                            h->stream) != cudaSuccess)
            return LLM_ERR_CUDA;
    }
    int rc = run_step(h);
    if (rc != LLM_OK) return rc;
    rc = fetch_token(h, out_token);
    if (rc != LLM_OK) return rc;
    h->seq_len += 1;
    h->have_token = true;
    h->stepped = true;
    return LLM_OK;
}

int llm_decode_enqueue(llm_t *h, int32_t n) {
    if (!h || n < 0) return LLM_ERR_ARG;
    if (n > 0 && !h->have_token) return LLM_ERR_STATE;
    if ((int64_t)h->seq_len + n > h->cfg.max_context) return LLM_ERR_CONTEXT_FULL;
    for (int i = 0; i < n; ++i) {
        int rc = run_step(h);
        if (rc != LLM_OK) return rc;
        h->seq_len += 1;
    }
    if (n > 0) h->stepped = true;
    return LLM_OK;
}

int llm_sync(llm_t *h) {
    if (!h) return LLM_ERR_ARG;
    return fetch_token(h, nullptr);
}

int llm_last_token(llm_t *h, int32_t *token) {
    if (!h || !token) return LLM_ERR_ARG;
    if (!h->stepped) return LLM_ERR_STATE;
    return fetch_token(h, token);
}

int llm_logits(llm_t *h, float *host_out, int32_t vocab) {
    if (!h || !host_out || vocab != h->cfg.vocab) return LLM_ERR_ARG;
    if (!h->stepped) return LLM_ERR_STATE;
    if (cudaMemcpyAsync(host_out, h->logits, (size_t)vocab * sizeof(float), cudaMemcpyDeviceToHost,
                        h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    return cudaStreamSynchronize(h->stream) == cudaSuccess ? LLM_OK : LLM_ERR_CUDA;
}

int llm_seq_len(llm_t *h, int32_t *seq_len) {
    if (!h || !seq_len) return LLM_ERR_ARG;
    *seq_len = h->seq_len;
    return LLM_OK;
}

int llm_reset(llm_t *h) {
    if (!h) return LLM_ERR_ARG;
    k_set_state<<<1, 1, 0, h->stream>>>(h->st, -1, 0, 1);
    if (cudaGetLastError() != cudaSuccess) return LLM_ERR_CUDA;
    // a step that failed part-way leaves its counters raised
    if (h->step_sync && cudaMemsetAsync(h->step_sync, 0, ((size_t)h->cfg.n_layers * kSyncStride + 1) * sizeof(int),
                                        h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    // ... and a part-way o_proj fold output
    if (h->o_d && cudaMemsetAsync(h->o_d, 0, (size_t)h->cfg.hidden * sizeof(long long), h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
    h->seq_len = 0;
    h->have_token = false;
    h->stepped = false;
    return LLM_OK;
}

int llm_truncate(llm_t *h, int32_t seq_len) {
    if (!h || seq_len < 0 || seq_len > h->seq_len) return LLM_ERR_ARG;
    k_set_state<<<1, 1, 0, h->stream>>>(h->st, -1, seq_len, 0);
    if (cudaGetLastError() != cudaSuccess) return LLM_ERR_CUDA;
    h->seq_len = seq_len;
    return LLM_OK;
}

int llm_timeline_steps(llm_t *h, int32_t n_steps, uint64_t *stamps, int32_t cap, int32_t *n_per_step) {
    if (!h || n_steps < 1 || !stamps || !n_per_step) return LLM_ERR_ARG;
    if (h->persistent || !h->have_token) return h->persistent ? LLM_ERR_ARG : LLM_ERR_STATE;
    if ((int64_t)h->seq_len + n_steps > h->cfg.max_context) return LLM_ERR_CONTEXT_FULL;
    const int per = 5 * h->cfg.n_layers + 2;  // upper bound on launches per step
    if ((int64_t)cap < (int64_t)n_steps * per) return LLM_ERR_ARG;
    unsigned long long *tl = nullptr;
    const size_t bytes = (size_t)n_steps * per * sizeof(unsigned long long);
    if (cudaStreamSynchronize(h->stream) != cudaSuccess || cudaMalloc((void **)&tl, bytes) != cudaSuccess)
        return LLM_ERR_CUDA;
    cudaGraph_t g = nullptr;
    cudaGraphExec_t x = nullptr;
    int rc = LLM_OK, n = 0;
    if (cudaMemsetAsync(tl, 0, bytes, h->stream) != cudaSuccess ||
        cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
        rc = LLM_ERR_CUDA;
    } else {
        cudaError_t ce = cudaSuccess;
        for (int i = 0; i < n_steps && ce == cudaSuccess; ++i) ce = enqueue_step(h, nullptr, tl + (size_t)i * per, &n);
        cudaError_t ee = cudaStreamEndCapture(h->stream, &g);
        if (ce != cudaSuccess || ee != cudaSuccess || cudaGraphInstantiate(&x, g, 0) != cudaSuccess ||
            cudaGraphLaunch(x, h->stream) != cudaSuccess)
            rc = LLM_ERR_CUDA;
    }
    if (rc == LLM_OK) {
        rc = fetch_token(h, nullptr);
        if (rc == LLM_OK) {
            h->seq_len += n_steps;
            h->stepped = true;
            std::vector<unsigned long long> host((size_t)n_steps * per);
            if (cudaMemcpy(host.data(), tl, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
                rc = LLM_ERR_CUDA;
            } else {
                for (int i = 0; i < n_steps; ++i)
                    for (int j = 0; j < n; ++j) stamps[(size_t)i * n + j] = host[(size_t)i * per + j];
                *n_per_step = n;
            }
        }
    }
    if (x) cudaGraphExecDestroy(x);
    if (g) cudaGraphDestroy(g);
    cudaFree(tl);
    return rc;
}

int llm_profile_step(llm_t *h, float *kernel_ms, int32_t cap, int32_t *n_kernels) {
    if (!h || !kernel_ms || !n_kernels) return LLM_ERR_ARG;
    const int n = 5 * h->cfg.n_layers + 1;
    *n_kernels = n;
    if (cap < n) return LLM_ERR_ARG;
    if (!h->have_token) return LLM_ERR_STATE;
    if (h->seq_len >= h->cfg.max_context) return LLM_ERR_CONTEXT_FULL;
    if (h->persistent) {
        StepParams p = h->sp;
        p.prof = h->prof;
        std::vector<unsigned long long> ts((size_t)n + 1);
        if (cudaMemsetAsync(h->prof, 0, ts.size() * sizeof(unsigned long long), h->stream) != cudaSuccess ||
            launch_step(h->sl, p, h->stream) != cudaSuccess ||
            cudaMemcpyAsync(ts.data(), h->prof, ts.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost,
                            h->stream) != cudaSuccess ||
            cudaStreamSynchronize(h->stream) != cudaSuccess)
            return LLM_ERR_CUDA;
        int rc = fetch_token(h, nullptr);
        if (rc != LLM_OK) return rc;
        for (int i = 0; i < n; ++i)
            kernel_ms[i] = ts[i + 1] >= ts[i] ? (float)((double)(ts[i + 1] - ts[i]) * 1e-6) : 0.f;
        h->seq_len += 1;
        h->stepped = true;
        return LLM_OK;
    }
    std::vector<cudaEvent_t> ev(n + 1, nullptr);
    int rc = LLM_OK;
    for (auto &e : ev)
        if (cudaEventCreate(&e) != cudaSuccess) rc = LLM_ERR_CUDA;
    if (rc == LLM_OK) {
        const bool pdl = h->lc.pdl;
        h->lc.pdl = false;
        cudaError_t e = enqueue_step(h, ev.data());
        h->lc.pdl = pdl;
        if (e != cudaSuccess || cudaStreamSynchronize(h->stream) != cudaSuccess) rc = LLM_ERR_CUDA;
    }
    for (int i = 0; rc == LLM_OK && i < n; ++i)
        if (cudaEventElapsedTime(&kernel_ms[i], ev[i], ev[i + 1]) != cudaSuccess) rc = LLM_ERR_CUDA;
    for (auto &e : ev)
        if (e) cudaEventDestroy(e);
    if (rc != LLM_OK) return rc;
    rc = fetch_token(h, nullptr);
    if (rc != LLM_OK) return rc;
    h->seq_len += 1;
    h->stepped = true;
    return LLM_OK;
}

int llm_debug_kv(llm_t *h, void **k_pool, void **v_pool, int32_t **page_table, int32_t *n_pages,
                 int32_t set_len) {
    if (!h) return LLM_ERR_ARG;
    if (set_len > h->cfg.max_context) return LLM_ERR_ARG;
    if (k_pool) *k_pool = h->k_pool;
    if (v_pool) *v_pool = h->v_pool;
    if (page_table) *page_table = h->page_table;
    if (n_pages) *n_pages = h->n_pages;
    if (set_len >= 0) {
        k_set_state<<<1, 1, 0, h->stream>>>(h->st, -1, set_len, 0);
        if (cudaGetLastError() != cudaSuccess) return LLM_ERR_CUDA;
        if (cudaStreamSynchronize(h->stream) != cudaSuccess) return LLM_ERR_CUDA;
        h->seq_len = set_len;
    }
    return LLM_OK;
}

}  // extern "C"
