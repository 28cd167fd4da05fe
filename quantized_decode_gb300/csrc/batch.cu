// batch.cu - multi-sequence decode behind llm_batch_* (llm.h).
//
// Up to 8 sequences share one engine: one K/V pool of 16-token pages
// [L][pages][Hkv][16][d] handed out by a host-side allocator (a free list; page 0
// is reserved and never handed out), a page table and a device state (position,
// input token, last token, error word) per sequence slot ("Systems Foundations
// for LLMs", PagedAttention and its block manager: per-sequence block tables,
// blocks taken on demand and returned when a sequence ends).  A step runs every
// slot through the layers at once: the linear layers as skinny GEMMs on the
// tensor cores that read each weight once for all slots (k_batch.cu), attention
// per sequence with that sequence's page table and length (the split-K kernel of
// the single-sequence engine), and a greedy argmax per sequence.  Slots that do
// not take part in a step (free, or not asked for) compute on stale inputs, but
// write no K/V and keep their position; a free slot's page table points at the
// reserved page.  The step is captured once into a CUDA graph; which slots take
// part, and their forced inputs, are device data written before each replay.
#include <algorithm>
#include <cmath>
#include <new>
#include <vector>

#include "../../include/llm.h"
#include "kernels.h"

using namespace qd;

struct llm_batch_t {
    llm_config cfg;
    int fmt = 0;
    std::vector<llm_layer_weights> layers;
    llm_weights w{};
    cudaStream_t stream = nullptr;
    bool own_stream = false;
    LaunchCfg lc{};
    int S = 0;                    // sequence slots
    int n_pages = 0, max_pages = 0;
    size_t layer_kv = 0;          // elements of one layer's pool
    uint16_t *k_pool = nullptr, *v_pool = nullptr;
    int *page_table = nullptr;    // [S][max_pages]
    DevState *st = nullptr;       // [S]
    int *part = nullptr;          // [S]
    float2 *rope_cs = nullptr;
    float *x = nullptr, *raw = nullptr, *q = nullptr, *attn = nullptr, *u = nullptr, *logits = nullptr;
    float *part_o = nullptr, *part_ml = nullptr;  // per slot: attention split partials
    int *attn_cnt = nullptr;                      // per slot: arrival counters
    float *arg_v = nullptr;                       // split argmax scratch [S][32]
    int *arg_i = nullptr;
    std::vector<cudaStream_t> side;               // per slot: the attention branch of the graph
    std::vector<cudaEvent_t> ev;                  // fork event, then one join event per slot
    int P = 8, cs = 8;
    int32_t *pinned = nullptr;    // host staging: part [S] | state in [S] | state out [S] | page table [S][max_pages]
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    // host mirror
    std::vector<int> free_pages;  // popped from the back
    std::vector<std::vector<int>> pages;  // per slot: physical pages in logical order
    std::vector<int> len;         // per slot: tokens in the cache
    std::vector<char> live;       // per slot: holds a sequence
    std::vector<char> has_token;  // per slot: a previous step emitted a token to feed
    std::vector<int> last;        // per slot: the token the last step emitted

    int32_t *h_part() { return pinned; }
    DevState *h_st_in() { return reinterpret_cast<DevState *>(pinned + S); }
    DevState *h_st_out() { return reinterpret_cast<DevState *>(pinned + S + 4 * S); }
    int32_t *h_ptab() { return pinned + S + 8 * S; }
};

int engine_validate(const llm_config *c, const llm_weights *w);  // engine.cu

namespace {

template <typename T>
cudaError_t dalloc(T **p, size_t n) {
    return cudaMalloc(reinterpret_cast<void **>(p), n * sizeof(T));
}

void free_all(llm_batch_t *h) {
    if (h->exec) cudaGraphExecDestroy(h->exec);
    if (h->graph) cudaGraphDestroy(h->graph);
    void *bufs[] = {h->k_pool, h->v_pool, h->page_table, h->st, h->part, h->rope_cs, h->x, h->raw, h->q,
                    h->attn, h->u, h->logits, h->part_o, h->part_ml, h->attn_cnt, h->arg_v, h->arg_i};
    for (void *b : bufs)
        if (b) cudaFree(b);
    if (h->pinned) cudaFreeHost(h->pinned);
    for (cudaStream_t x : h->side)
        if (x) cudaStreamDestroy(x);
    for (cudaEvent_t e : h->ev)
        if (e) cudaEventDestroy(e);
    if (h->own_stream && h->stream) cudaStreamDestroy(h->stream);
}

cudaError_t enqueue_batch_step(llm_batch_t *h) {
    const llm_config &c = h->cfg;
    const int d = c.head_dim, rq = c.n_q_heads * d, rkv = c.n_kv_heads * d, nq = rq + 2 * rkv, S = h->S;
    cudaError_t e = launch_bembed(h->stream, (const uint16_t *)h->w.embed, h->st, S, c.hidden, h->x);
    if (e != cudaSuccess) return e;
    for (int l = 0; l < c.n_layers; ++l) {
        const llm_layer_weights &L = h->layers[l];
        uint16_t *kp = h->k_pool + (size_t)l * h->layer_kv, *vp = h->v_pool + (size_t)l * h->layer_kv;
        BGemvArgs g{};
        g.mode = 0; g.n_seg = 3;
        g.w[0] = L.wq; g.w[1] = L.wk; g.w[2] = L.wv;
        g.s[0] = L.sq; g.s[1] = L.sk; g.s[2] = L.sv;
        if (c.qkv_bias) {
            g.bias[0] = (const uint16_t *)L.bq; g.bias[1] = (const uint16_t *)L.bk; g.bias[2] = (const uint16_t *)L.bv;
        }
        g.seg_rows[0] = rq; g.seg_rows[1] = rkv; g.seg_rows[2] = rkv;
        g.N = nq; g.K = c.hidden; g.B = S; g.x = h->x; g.ldx = c.hidden;
        g.gamma = (const uint16_t *)L.attn_norm; g.eps = c.rms_eps; g.y = h->raw; g.ldy = nq;
        if ((e = launch_bgemv(h->lc, h->fmt, g)) != cudaSuccess) return e;

        BQkvPostArgs pa{};
        pa.raw = h->raw; pa.Hq = c.n_q_heads; pa.Hkv = c.n_kv_heads; pa.d = d;
        if (c.qk_norm) {
            pa.q_gain = (const uint16_t *)L.q_norm;
            pa.k_gain = (const uint16_t *)L.k_norm;
        }
        pa.eps = c.rms_eps; pa.rope_cs = h->rope_cs; pa.q_out = h->q; pa.k_pool = kp; pa.v_pool = vp;
        pa.page_table = h->page_table; pa.max_pages = h->max_pages; pa.n_pages = h->n_pages;
        pa.st = h->st; pa.part = h->part;
        if ((e = launch_bqkv_post(h->stream, pa, S)) != cudaSuccess) return e;

        // attention per sequence, through its own table and length: one graph branch
        // per sequence (its own stream while capturing), so they run side by side
        const int G = c.n_q_heads / c.n_kv_heads;
        if ((e = cudaEventRecord(h->ev[0], h->stream)) != cudaSuccess) return e;
        for (int b = 0; b < S; ++b) {
            if ((e = cudaStreamWaitEvent(h->side[b], h->ev[0], 0)) != cudaSuccess) return e;
            LaunchCfg lb = h->lc;
            lb.stream = h->side[b];
            AttnArgs aa{};
            aa.q = h->q + (size_t)b * rq;
            aa.k_pool = kp; aa.v_pool = vp;
            aa.page_table = h->page_table + (size_t)b * h->max_pages; aa.n_pages = h->n_pages;
            aa.st = h->st + b; aa.T_fixed = -1;
            aa.Hq = c.n_q_heads; aa.Hkv = c.n_kv_heads; aa.d = d; aa.P = h->P; aa.cs = h->cs;
            aa.part_o = h->part_o + (size_t)b * c.n_kv_heads * h->P * G * d;
            aa.part_ml = h->part_ml + (size_t)b * c.n_kv_heads * h->P * G * 2;
            aa.counter = h->attn_cnt + (size_t)b * c.n_kv_heads;
            aa.out = h->attn + (size_t)b * rq; aa.err = &h->st[b].err;
            if ((e = launch_attention(lb, aa)) != cudaSuccess) return e;
            if ((e = cudaEventRecord(h->ev[1 + b], h->side[b])) != cudaSuccess) return e;
        }
        for (int b = 0; b < S; ++b)
            if ((e = cudaStreamWaitEvent(h->stream, h->ev[1 + b], 0)) != cudaSuccess) return e;

        BGemvArgs o{};
        o.mode = 1; o.n_seg = 1; o.w[0] = L.wo; o.s[0] = L.so; o.seg_rows[0] = c.hidden;
        o.N = c.hidden; o.K = rq; o.B = S; o.x = h->attn; o.ldx = rq; o.y = h->x; o.ldy = c.hidden;
        if ((e = launch_bgemv(h->lc, h->fmt, o)) != cudaSuccess) return e;

        BGemvArgs gu{};
        gu.mode = 2; gu.n_seg = 1; gu.w[0] = L.wg; gu.s[0] = L.sg; gu.w2 = L.wu; gu.s2 = L.su;
        gu.N = c.mlp; gu.K = c.hidden; gu.B = S; gu.x = h->x; gu.ldx = c.hidden;
        gu.gamma = (const uint16_t *)L.mlp_norm; gu.eps = c.rms_eps; gu.y = h->u; gu.ldy = c.mlp;
        if ((e = launch_bgemv(h->lc, h->fmt, gu)) != cudaSuccess) return e;

        BGemvArgs dn{};
        dn.mode = 1; dn.n_seg = 1; dn.w[0] = L.wd; dn.s[0] = L.sd; dn.seg_rows[0] = c.hidden;
        dn.N = c.hidden; dn.K = c.mlp; dn.B = S; dn.x = h->u; dn.ldx = c.mlp; dn.y = h->x; dn.ldy = c.hidden;
        if ((e = launch_bgemv(h->lc, h->fmt, dn)) != cudaSuccess) return e;
    }
    const bool int8_head = h->fmt == kFmtInt8 && !c.tied_lm_head;
    BGemvArgs lm{};
    lm.mode = 3; lm.n_seg = 1;
    lm.w[0] = c.tied_lm_head ? h->w.embed : h->w.lm_head;
    lm.s[0] = int8_head ? h->w.lm_scale : nullptr;
    lm.seg_rows[0] = c.vocab;
    lm.N = c.vocab; lm.K = c.hidden; lm.B = S; lm.x = h->x; lm.ldx = c.hidden;
    lm.gamma = (const uint16_t *)h->w.final_norm; lm.eps = c.rms_eps; lm.y = h->logits; lm.ldy = c.vocab;
    if ((e = launch_bgemv(h->lc, int8_head ? kFmtInt8 : kFmtBf16, lm)) != cudaSuccess) return e;
    return launch_bargmax(h->stream, h->logits, c.vocab, h->st, S, h->part, h->arg_v, h->arg_i);
}

int capture(llm_batch_t *h) {
    if (cudaStreamBeginCapture(h->stream, cudaStreamCaptureModeThreadLocal) != cudaSuccess) return LLM_ERR_CUDA;
    cudaError_t ce = enqueue_batch_step(h);
    cudaError_t ee = cudaStreamEndCapture(h->stream, &h->graph);
    if (ce != cudaSuccess || ee != cudaSuccess) return LLM_ERR_CUDA;
    return cudaGraphInstantiate(&h->exec, h->graph, 0) == cudaSuccess ? LLM_OK : LLM_ERR_CUDA;
}

// Write slot b's page table entry i (pinned mirror, then the device copy), stream-ordered.
int set_page(llm_batch_t *h, int b, int i, int page) {
    int32_t *m = h->h_ptab() + (size_t)b * h->max_pages + i;
    *m = page;
    return cudaMemcpyAsync(h->page_table + (size_t)b * h->max_pages + i, m, sizeof(int), cudaMemcpyHostToDevice,
                           h->stream) == cudaSuccess
               ? LLM_OK
               : LLM_ERR_CUDA;
}

}  // namespace

extern "C" {

int llm_batch_create(const llm_config *cfg, const llm_weights *w, int32_t max_seqs, int32_t n_pages,
                     void *cuda_stream, llm_batch_t **out) {
    if (!out) return LLM_ERR_ARG;
    *out = nullptr;
    if (!cfg || !w || !w->layers || max_seqs < 1 || max_seqs > 8 || n_pages < 0) return LLM_ERR_ARG;
    // the single-sequence engine's validation (shapes, alignment, layout id)
    int rc = engine_validate(cfg, w);
    if (rc != LLM_OK) return rc;
    const int fmt = cfg->weight_format == LLM_FMT_INT4_G128 ? kFmtInt4 : kFmtInt8;
    const int d = cfg->head_dim, rq = cfg->n_q_heads * d, rkv = cfg->n_kv_heads * d;
    const bool int8_head = fmt == kFmtInt8 && !cfg->tied_lm_head;
    if (!bgemv_shape_ok(fmt, rq + 2 * rkv, cfg->hidden, 0) || !bgemv_shape_ok(fmt, cfg->hidden, rq, 1) ||
        !bgemv_shape_ok(fmt, cfg->mlp, cfg->hidden, 2) || !bgemv_shape_ok(fmt, cfg->hidden, cfg->mlp, 1) ||
        !bgemv_shape_ok(int8_head ? kFmtInt8 : kFmtBf16, cfg->vocab, cfg->hidden, 3) || rq % 16 || rkv % 16)
        return LLM_ERR_ARG;

    llm_batch_t *h = new (std::nothrow) llm_batch_t();
    if (!h) return LLM_ERR_CUDA;
    auto fail = [&](int code) {
        free_all(h);
        delete h;
        return code;
    };
    h->cfg = *cfg;
    h->fmt = fmt;
    h->layers.assign(w->layers, w->layers + cfg->n_layers);
    h->w = *w;
    h->w.layers = nullptr;
    h->S = max_seqs;
    int dev = 0, n_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(LLM_ERR_CUDA);
    if (cuda_stream) {
        h->stream = (cudaStream_t)cuda_stream;
    } else {
        if (cudaStreamCreateWithFlags(&h->stream, cudaStreamNonBlocking) != cudaSuccess) return fail(LLM_ERR_CUDA);
        h->own_stream = true;
    }
    h->lc.stream = h->stream;
    h->lc.pdl = true;  // the GEMMs and the attention wait for their predecessor before touching activations
    h->lc.n_sm = n_sm;
    const llm_config &c = h->cfg;
    h->max_pages = (c.max_context + kPageTokens - 1) / kPageTokens;
    h->n_pages = n_pages > 0 ? n_pages : max_seqs * h->max_pages + 1;
    if (h->n_pages < 2 || (int64_t)h->n_pages * c.n_kv_heads * kPageTokens > INT32_MAX) return fail(LLM_ERR_ARG);
    h->layer_kv = (size_t)h->n_pages * c.n_kv_heads * kPageTokens * d;
    AttnPlan ap = plan_attention(n_sm, c.n_q_heads, c.n_kv_heads, d, h->max_pages);
    // the sequences' attention kernels run side by side: narrower clusters, one cluster per KV
    // head and sequence, once max_seqs of the single-sequence plan would take more than the SMs
    if ((long long)max_seqs * c.n_kv_heads * ap.P > n_sm) {
        const int cs = (long long)max_seqs * c.n_kv_heads * 8 <= n_sm ? 8 : 4;
        ap = AttnPlan{cs, cs};
    }
    h->P = ap.P;
    h->cs = ap.cs;
    const int G = c.n_q_heads / c.n_kv_heads;
    const int nq = rq + 2 * rkv, S = max_seqs;
    bool ok = dalloc(&h->k_pool, h->layer_kv * c.n_layers) == cudaSuccess &&
              dalloc(&h->v_pool, h->layer_kv * c.n_layers) == cudaSuccess &&
              dalloc(&h->page_table, (size_t)S * h->max_pages) == cudaSuccess && dalloc(&h->st, S) == cudaSuccess &&
              dalloc(&h->part, S) == cudaSuccess &&
              dalloc(&h->rope_cs, (size_t)c.max_context * (d / 2)) == cudaSuccess &&
              dalloc(&h->x, (size_t)S * c.hidden) == cudaSuccess && dalloc(&h->raw, (size_t)S * nq) == cudaSuccess &&
              dalloc(&h->q, (size_t)S * rq) == cudaSuccess && dalloc(&h->attn, (size_t)S * rq) == cudaSuccess &&
              dalloc(&h->u, (size_t)S * c.mlp) == cudaSuccess && dalloc(&h->logits, (size_t)S * c.vocab) == cudaSuccess &&
              dalloc(&h->part_o, (size_t)S * c.n_kv_heads * h->P * G * d) == cudaSuccess &&
              dalloc(&h->part_ml, (size_t)S * c.n_kv_heads * h->P * G * 2) == cudaSuccess &&
              dalloc(&h->attn_cnt, (size_t)S * c.n_kv_heads) == cudaSuccess &&
              dalloc(&h->arg_v, (size_t)S * 32) == cudaSuccess && dalloc(&h->arg_i, (size_t)S * 32) == cudaSuccess &&
              cudaMallocHost((void **)&h->pinned, sizeof(int32_t) * ((size_t)S * 9 + (size_t)S * h->max_pages)) ==
                  cudaSuccess;
    h->side.assign(S, nullptr);
    h->ev.assign(S + 1, nullptr);
    for (int b = 0; ok && b < S; ++b)
        ok = cudaStreamCreateWithFlags(&h->side[b], cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; ok && i <= S; ++i) ok = cudaEventCreateWithFlags(&h->ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) return fail(LLM_ERR_CUDA);
    ok = cudaMemsetAsync(h->page_table, 0, sizeof(int) * (size_t)S * h->max_pages, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->st, 0, sizeof(DevState) * S, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->part, 0, sizeof(int) * S, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->attn_cnt, 0, sizeof(int) * (size_t)S * c.n_kv_heads, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->x, 0, sizeof(float) * (size_t)S * c.hidden, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->attn, 0, sizeof(float) * (size_t)S * rq, h->stream) == cudaSuccess &&
         cudaMemsetAsync(h->u, 0, sizeof(float) * (size_t)S * c.mlp, h->stream) == cudaSuccess;
    std::vector<float2> cs((size_t)c.max_context * (d / 2));
    for (int p = 0; p < c.max_context; ++p)
        for (int i = 0; i < d / 2; ++i) {
            const double ang = (double)p * std::pow((double)c.rope_base, -2.0 * (double)i / (double)d);
            cs[(size_t)p * (d / 2) + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
        }
    ok = ok && cudaMemcpyAsync(h->rope_cs, cs.data(), cs.size() * sizeof(float2), cudaMemcpyHostToDevice,
                               h->stream) == cudaSuccess &&
         cudaStreamSynchronize(h->stream) == cudaSuccess;
    if (!ok) return fail(LLM_ERR_CUDA);
    // free list: pages n_pages - 1 .. 1 (page 0 stays reserved), taken from the back
    for (int p = h->n_pages - 1; p >= 1; --p) h->free_pages.push_back(p);
    h->pages.assign(S, {});
    h->len.assign(S, 0);
    h->live.assign(S, 0);
    h->has_token.assign(S, 0);
    h->last.assign(S, 0);
    std::fill(h->pinned, h->pinned + (size_t)S * 9 + (size_t)S * h->max_pages, 0);
    if (capture(h) != LLM_OK) return fail(LLM_ERR_CUDA);
    *out = h;
    return LLM_OK;
}

void llm_batch_destroy(llm_batch_t *h) {
    if (!h) return;
    cudaStreamSynchronize(h->stream);
    free_all(h);
    delete h;
}

int llm_batch_add(llm_batch_t *h, int32_t *seq) {
    if (!h || !seq) return LLM_ERR_ARG;
    for (int b = 0; b < h->S; ++b)
        if (!h->live[b]) {
            h->live[b] = 1;
            h->len[b] = 0;
            h->has_token[b] = 0;
            h->pages[b].clear();
            *seq = b;
            return LLM_OK;
        }
    return LLM_ERR_STATE;
}

int llm_batch_release(llm_batch_t *h, int32_t seq) {
    if (!h || seq < 0 || seq >= h->S || !h->live[seq]) return LLM_ERR_ARG;
    // pages back on the free list; the slot's table entries point at the reserved page again
    for (int i = (int)h->pages[seq].size() - 1; i >= 0; --i) {
        h->free_pages.push_back(h->pages[seq][i]);
        if (set_page(h, seq, i, 0) != LLM_OK) return LLM_ERR_CUDA;
    }
    h->pages[seq].clear();
    h->live[seq] = 0;
    h->len[seq] = 0;
    h->has_token[seq] = 0;
    h->last[seq] = 0;
    return cudaStreamSynchronize(h->stream) == cudaSuccess ? LLM_OK : LLM_ERR_CUDA;
}

int llm_batch_set_page_order(llm_batch_t *h, const int32_t *order, int32_t n) {
    if (!h || !order || n != h->n_pages - 1) return LLM_ERR_ARG;
    for (int b = 0; b < h->S; ++b)
        if (h->live[b]) return LLM_ERR_STATE;
    std::vector<char> seen(h->n_pages, 0);
    for (int i = 0; i < n; ++i) {
        if (order[i] < 1 || order[i] >= h->n_pages || seen[order[i]]) return LLM_ERR_ARG;
        seen[order[i]] = 1;
    }
    h->free_pages.assign(order, order + n);
    std::reverse(h->free_pages.begin(), h->free_pages.end());  // order[0] is handed out first
    return LLM_OK;
}

int llm_batch_step(llm_batch_t *h, const int32_t *seqs, const int32_t *inputs, int32_t n, int32_t *out_tokens) {
    if (!h || !seqs || n < 1 || n > h->S) return LLM_ERR_ARG;
    const llm_config &c = h->cfg;
    std::vector<char> take(h->S, 0);
    for (int i = 0; i < n; ++i) {
        const int b = seqs[i];
        if (b < 0 || b >= h->S || !h->live[b] || take[b]) return LLM_ERR_ARG;
        if (inputs && inputs[i] >= c.vocab) return LLM_ERR_ARG;
        if ((!inputs || inputs[i] < 0) && !h->has_token[b]) return LLM_ERR_STATE;
        if (h->len[b] >= c.max_context) return LLM_ERR_CONTEXT_FULL;
        take[b] = 1;
    }
    // a page for every sequence that starts one now (before any launch: all or nothing)
    int need = 0;
    for (int i = 0; i < n; ++i)
        if (h->len[seqs[i]] % kPageTokens == 0) ++need;
    if (need > (int)h->free_pages.size()) return LLM_ERR_CONTEXT_FULL;
    for (int i = 0; i < n; ++i) {
        const int b = seqs[i];
        if (h->len[b] % kPageTokens == 0) {
            const int p = h->free_pages.back();
            h->free_pages.pop_back();
            h->pages[b].push_back(p);
            if (set_page(h, b, h->len[b] / kPageTokens, p) != LLM_OK) return LLM_ERR_CUDA;
        }
    }
    // every slot's state as the host holds it (the inputs of the sequences in this
    // step, their positions), the part flags, then one replay
    int32_t *part = h->h_part();
    DevState *sin = h->h_st_in(), *sout = h->h_st_out();
    for (int b = 0; b < h->S; ++b) {
        part[b] = take[b];
        sin[b].pos = h->live[b] ? h->len[b] : 0;
        sin[b].token = h->last[b];
        sin[b].last_token = h->last[b];
        sin[b].err = kErrNone;
    }
    for (int i = 0; i < n; ++i)
        if (inputs && inputs[i] >= 0) sin[seqs[i]].token = inputs[i];
    if (cudaMemcpyAsync(h->part, part, sizeof(int32_t) * h->S, cudaMemcpyHostToDevice, h->stream) != cudaSuccess ||
        cudaMemcpyAsync(h->st, sin, sizeof(DevState) * h->S, cudaMemcpyHostToDevice, h->stream) != cudaSuccess ||
        cudaGraphLaunch(h->exec, h->stream) != cudaSuccess ||
        cudaMemcpyAsync(sout, h->st, sizeof(DevState) * h->S, cudaMemcpyDeviceToHost, h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    for (int i = 0; i < n; ++i) {
        const int b = seqs[i];
        if (sout[b].err != kErrNone) return sout[b].err == kErrTimeout ? LLM_ERR_TIMEOUT : LLM_ERR_DEVICE;
    }
    for (int i = 0; i < n; ++i) {
        const int b = seqs[i];
        h->len[b] += 1;
        h->has_token[b] = 1;
        h->last[b] = sout[b].last_token;
        if (out_tokens) out_tokens[i] = sout[b].last_token;
    }
    return LLM_OK;
}

int llm_batch_prefill(llm_batch_t *h, int32_t seq, const int32_t *tokens, int32_t n, int32_t *first_token) {
    if (!h || !tokens || n < 1 || seq < 0 || seq >= h->S || !h->live[seq]) return LLM_ERR_ARG;
    if (h->len[seq] + n > h->cfg.max_context) return LLM_ERR_CONTEXT_FULL;
    int32_t out = 0;
    for (int i = 0; i < n; ++i) {
        if (tokens[i] < 0 || tokens[i] >= h->cfg.vocab) return LLM_ERR_ARG;
        int rc = llm_batch_step(h, &seq, &tokens[i], 1, &out);
        if (rc != LLM_OK) return rc;
    }
    if (first_token) *first_token = out;
    return LLM_OK;
}

int llm_batch_logits(llm_batch_t *h, int32_t seq, float *host_out, int32_t vocab) {
    if (!h || !host_out || vocab != h->cfg.vocab || seq < 0 || seq >= h->S || !h->live[seq]) return LLM_ERR_ARG;
    if (!h->has_token[seq]) return LLM_ERR_STATE;
    if (cudaMemcpyAsync(host_out, h->logits + (size_t)seq * vocab, sizeof(float) * vocab, cudaMemcpyDeviceToHost,
                        h->stream) != cudaSuccess ||
        cudaStreamSynchronize(h->stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    return LLM_OK;
}

int llm_batch_seq_info(llm_batch_t *h, int32_t seq, int32_t *len, int32_t *pages, int32_t cap, int32_t *n_pages,
                       int32_t *free_pages) {
    if (!h || seq < 0 || seq >= h->S) return LLM_ERR_ARG;
    if (len) *len = h->live[seq] ? h->len[seq] : 0;
    const int np = (int)h->pages[seq].size();
    if (n_pages) *n_pages = np;
    if (pages) {
        if (cap < np) return LLM_ERR_ARG;
        for (int i = 0; i < np; ++i) pages[i] = h->pages[seq][i];
    }
    if (free_pages) *free_pages = (int32_t)h->free_pages.size();
    return LLM_OK;
}

int llm_batch_debug_kv(llm_batch_t *h, void **k_pool, void **v_pool, int32_t *n_pages) {
    if (!h) return LLM_ERR_ARG;
    if (k_pool) *k_pool = h->k_pool;
    if (v_pool) *v_pool = h->v_pool;
    if (n_pages) *n_pages = h->n_pages;
    return LLM_OK;
}

}  // extern "C"
