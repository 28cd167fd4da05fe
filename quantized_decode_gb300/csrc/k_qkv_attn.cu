// k_qkv_attn.cu - QKV projection and decode attention of one layer in one kernel
// (models without per-head q/k norms, head_dim 128, one 16-CTA cluster per KV
// head).
//
// The cluster of KV head g owns the group's (G + 2) heads of projection rows:
// its G query heads, K head g and V head g, (G + 2) * 64 RoPE pairs, cut into
// tiles of 4 pairs of one head; CTA r of the cluster computes tiles
// r (G + 2) .. r (G + 2) + G + 1.  In order:
//   1. the CTA's projection weights go out before the dependency wait, the
//      whole slice at once: their ring (11 steps per warp) spans the shared
//      memory that the attention's page ring uses later;
//   2. after the wait: RMSNorm(x) staged, the weights consumed, and per tile the
//      warps' K parts summed, bias and RoPE applied; K and V of the new
//      position are rounded to bf16 and written to the page;
//   3. the CTA's K/V page copies go out (every page is final before the step
//      but the appended row, which comes from step 2), and meanwhile the
//      cluster exchanges the tiles through distributed shared memory: every
//      CTA gathers the group's queries and the new K/V row;
//   4. the split-K attention of attn.cuh over the CTA's pages, merged in the
//      cluster, writes the output rows and their statistics.
// Compared with a QKV kernel followed by an attention kernel, the step loses
// one kernel boundary (grid completion, launch, staging of the query); the
// 152 - 16 Hkv SMs that the clusters leave free take the next kernel's early
// CTAs, which prefetch its weights meanwhile.
#include "attn.cuh"
#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

using namespace attn;

constexpr int kD128 = 128;
constexpr int kQRT = 2;                // rows per lane: a RoPE pair (p, p + 64)
constexpr int kQD = 11;                // projection ring depth (10 steps in flight)
constexpr int kQLPR = kLanesPerRow;
constexpr int kQS = 32 / kQLPR;        // row slots per warp: 4 pairs per tile
constexpr int kTilesPerHead = kD128 / 2 / kQS;  // 16

// Dynamic shared memory: the projection rings, then (same bytes) the
// attention's page ring; after them, in order, the rest.
struct FusedLayout {
    size_t xs, rings, kred, rows, ep, q, kv, total;
};
QD_HOST_DEV_INLINE FusedLayout fused_layout(int G, int K) {
    FusedLayout L;
    const size_t proj = (size_t)kWarps * ring_bytes_per_warp<kQRT, kQD>();
    L.rings = 0;
    size_t o = ((proj > ring_bytes<kD128>() ? proj : ring_bytes<kD128>()) + 127) & ~(size_t)127;
    L.xs = o;
    o += ((size_t)K * 2 + 15) & ~(size_t)15;
    L.kred = o;
    o += (size_t)kWarps * 32 * kQRT * 4;
    L.rows = o;
    o += (((size_t)(G + 2) * kQS * kQRT * 4) + 15) & ~(size_t)15;
    L.ep = o;  // per tile row: bias, INT8 row scale; per pair: RoPE (cos, sin)
    o += (size_t)(G + 2) * kQS * (kQRT * 4 + kQRT * 4 + 8);
    L.q = o;
    o += (size_t)G * kD128 * 4;
    L.kv = o;
    o += (size_t)2 * kD128 * 2;
    L.total = o + 1024;  // alignment slack of the base
    return L;
}

template <int FMT, int G>
__global__ void __launch_bounds__(kNT, 1) k_qkv_attn(QkvArgs qa, const __grid_constant__ AttnArgs at) {
    TimelineMark timeline_mark{qa.tl};
    constexpr int D = kD128;
    constexpr int NT = G + 2;  // tiles per CTA
    extern __shared__ __align__(128) uint16_t smem_raw[];
    uint16_t *smem = align_ring(smem_raw);  // the page ring's TMA boxes want 1024-byte alignment
    __shared__ float red[64];
    cg::cluster_group cluster = cg::this_cluster();
    const int g = blockIdx.y, rank = (int)cluster.block_rank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / kQLPR, j = lane % kQLPR;
    const FusedLayout L = fused_layout(G, qa.K);
    char *base = reinterpret_cast<char *>(smem);
    half2 *xs = reinterpret_cast<half2 *>(base + L.xs);
    float *kred = reinterpret_cast<float *>(base + L.kred);
    float *s_rows = reinterpret_cast<float *>(base + L.rows);  // [tile][slot][i]
    float *s_bias = reinterpret_cast<float *>(base + L.ep);    // [tile][slot][i]
    float *s_rsc = s_bias + NT * kQS * kQRT;                   // [tile][slot][i] (INT8)
    float2 *s_cs = reinterpret_cast<float2 *>(s_rsc + NT * kQS * kQRT);  // [tile][slot]
    float *s_q = reinterpret_cast<float *>(base + L.q);         // [G][D]
    uint16_t *s_kv = reinterpret_cast<uint16_t *>(base + L.kv); // [2][D] bf16

    auto hook = [&](auto &&issue_pages) -> AttnInputs {
        // ---- 2. projection rows of this CTA: the 8 warps form 8 / ks tile slots of
        // ks warps, each summing a non-empty part of K (ks <= slabs per row)
        uint4 *ring;
        uint32_t *sring;
        warp_rings<kQRT, kQD>(base + L.rings, kWarps, warp, ring, sring);
        const int NP = slabs_per_row(FMT, qa.K);
        const int U = units_per_row(FMT, qa.K);
        const int ks = NP >= 8 ? 8 : (NP >= 4 ? 4 : (NP >= 2 ? 2 : 1));
        const int tpc = kWarps / ks, kp = warp % ks, tslot = warp / ks;
        const int p_begin = kp * NP / ks, p_end = (kp + 1) * NP / ks;
        const size_t rb = FMT == kFmtInt4 ? (size_t)qa.K / 2 : (size_t)qa.K;
        const int Gs = qa.K / kGroup;
        float post = 1.f;
        int pos = 0, phys = -1;
        // tile t of this CTA: head hl of the group (G queries, then K, then V), pairs pp0 .. pp0 + 3
        auto tile_head = [&](int t) { return (rank * NT + t) / kTilesPerHead; };
        auto tile_pair = [&](int t) { return ((rank * NT + t) % kTilesPerHead) * kQS; };
        auto seg_row = [&](int hl, int row_in_head, int &seg) -> int {
            seg = hl < G ? 0 : (hl == G ? 1 : 2);
            return (hl < G ? (g * G + hl) : g) * D + row_in_head;
        };
        auto rows = [&](int t, int i) -> RowRef {
            int seg;
            const int r = seg_row(tile_head(t), tile_pair(t) + slot + i * (D / 2), seg);
            return {reinterpret_cast<const uint4 *>((const char *)qa.w[seg] + (size_t)r * rb),
                    (const uint16_t *)qa.s[seg] + (size_t)r * Gs};
        };
        auto sync = [&]() {
            // the tiles' epilogue constants, static data read before the wait (the
            // position is final too: the step's first kernel starts after the last step)
            pos = __ldcg(&qa.st->pos);
            for (int e = threadIdx.x; e < NT * kQS * kQRT; e += blockDim.x) {
                const int t = e / (kQS * kQRT), sl = (e / kQRT) % kQS, i = e % kQRT;
                int seg;
                const int r = seg_row(tile_head(t), tile_pair(t) + sl + i * (D / 2), seg);
                s_bias[e] = qa.b[seg] ? bf16_bits_to_float(__ldg(qa.b[seg] + r)) : 0.f;
                s_rsc[e] = FMT == kFmtInt8 ? __ldg((const float *)qa.s[seg] + r) : 1.f;
                if (i == 0) {
                    const int hl = tile_head(t);
                    s_cs[e / kQRT] = hl <= G ? __ldg(qa.rope_cs + (size_t)pos * (D / 2) + tile_pair(t) + sl)
                                             : make_float2(1.f, 0.f);
                }
            }
            phys = __ldg(qa.page_table + pos / kPageTokens);
            pdl_wait();
            const uint16_t *erow = qa.embed ? qa.embed + (size_t)__ldcg(&qa.st->token) * qa.K : nullptr;
            if (erow && g == 0 && rank == 0)
                for (int i = threadIdx.x; i < qa.K; i += blockDim.x) qa.x_init[i] = bf16_bits_to_float(erow[i]);
            post = stage_activations(qa.x, erow, qa.gamma, qa.eps, qa.K, erow ? nullptr : qa.stats_in, xs, nullptr,
                                     red, act_blk_bytes<FMT>(), nullptr, nullptr, nullptr, nullptr,
                                     erow ? nullptr : qa.x2);  // its barriers publish the constants
            pdl_launch();
        };
        auto epi = [&](int t, float(&out)[kQRT]) {
            if (!ksplit_reduce<kQRT>(out, ks, kp, tslot, kred + (size_t)tslot * ks * 32 * kQRT, j, slot, kQLPR) ||
                j != 0)
                return;
            const int hl = tile_head(t), p = tile_pair(t) + slot;
            const int seg = hl < G ? 0 : (hl == G ? 1 : 2);
            const int e = (t * kQS + slot) * kQRT;
            float v0 = out[0] * post, v1 = out[1] * post;
            if constexpr (FMT == kFmtInt8) {
                v0 *= s_rsc[e];
                v1 *= s_rsc[e + 1];
            }
            v0 += s_bias[e];
            v1 += s_bias[e + 1];
            if (seg < 2) {  // RoPE on q and k
                const float2 c = s_cs[t * kQS + slot];
                const float x0 = v0, x1 = v1;
                v0 = x0 * c.x - x1 * c.y;
                v1 = x1 * c.x + x0 * c.y;
            }
            s_rows[(t * kQS + slot) * kQRT] = v0;
            s_rows[(t * kQS + slot) * kQRT + 1] = v1;
            if (seg > 0) {  // the new K or V row into its page slot
                if (phys < 0 || phys >= qa.n_pages) {
                    atomicCAS(&qa.st->err, kErrNone, kErrBadPage);
                    return;
                }
                uint16_t *dst = (seg == 1 ? qa.k_pool : qa.v_pool) +
                                (((size_t)phys * qa.Hkv + g) * kPageTokens + pos % kPageTokens) * D;
                dst[p] = float_to_bf16_bits(v0);
                dst[p + D / 2] = float_to_bf16_bits(v1);
            }
        };
        gemv_stream<FMT, kQRT, kQD>(rows, epi, sync, tslot, tpc, NT, p_begin, p_end, U, j, xs, ring, sring);

        // ---- 3. every warp is done with the projection rings: the page copies
        // take their shared memory while the cluster exchanges the rows
        __syncthreads();
        issue_pages();
        cluster.sync();
        for (int idx = threadIdx.x; idx < (G + 2) * D; idx += blockDim.x) {
            const int hl = idx / D, dim = idx % D;
            const int pp = dim % (D / 2), i = dim / (D / 2);
            const int T = hl * kTilesPerHead + pp / kQS;
            const float *src = cluster.map_shared_rank(s_rows, T / NT);
            const float v = src[((T % NT) * kQS + pp % kQS) * kQRT + i];
            if (hl < G)
                s_q[hl * D + dim] = v;
            else
                s_kv[(hl - G) * D + dim] = float_to_bf16_bits(v);
        }
        __syncthreads();
        return AttnInputs{s_q, s_kv, s_kv + D};
    };
    // ---- 4: attn_cta runs the hook (1-3), then the attention
    attn_cta<G, D, kCSWide, true, true>(at, smem, hook);
}

template <int FMT, int G>
cudaError_t launch_fg(const LaunchCfg &lc, const QkvArgs &qa, const AttnArgs &at) {
    const FusedLayout L = fused_layout(G, qa.K);
    if (L.total > kMaxSmemOptin - 8 * 1024) return cudaErrorInvalidValue;  // static shared memory on top
    if (!allow_wide(k_qkv_attn<FMT, G>)) return cudaErrorInvalidValue;
    return launch_kc(lc, k_qkv_attn<FMT, G>, dim3(kCSWide, at.Hkv), dim3(kNT), L.total, kCSWide, qa, at);
}

template <int FMT>
cudaError_t launch_f(const LaunchCfg &lc, const QkvArgs &qa, const AttnArgs &at) {
    switch (at.Hq / at.Hkv) {
        case 1: return launch_fg<FMT, 1>(lc, qa, at);
        case 2: return launch_fg<FMT, 2>(lc, qa, at);
        case 3: return launch_fg<FMT, 3>(lc, qa, at);
        case 4: return launch_fg<FMT, 4>(lc, qa, at);
        case 5: return launch_fg<FMT, 5>(lc, qa, at);
        case 6: return launch_fg<FMT, 6>(lc, qa, at);
        case 7: return launch_fg<FMT, 7>(lc, qa, at);
        case 8: return launch_fg<FMT, 8>(lc, qa, at);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool qkv_attn_fusable(int fmt, int Hq, int Hkv, int d, int K, bool qk_norm, const AttnPlan &plan) {
    if (qk_norm || d != kD128 || plan.cs != kCSWide || plan.P != kCSWide) return false;
    if (fmt != kFmtInt4 && fmt != kFmtInt8) return false;
    if (Hkv < 1 || Hq % Hkv || Hq / Hkv > kMaxGqa) return false;
    if (fmt == kFmtInt4 ? (K % 256 != 0) : (K % 128 != 0)) return false;
    return fused_layout(Hq / Hkv, K).total <= kMaxSmemOptin - 8 * 1024;
}

cudaError_t launch_qkv_attn(const LaunchCfg &lc, int fmt, const QkvArgs &qa, const AttnArgs &args) {
    if (args.P != kCSWide || args.cs != kCSWide || args.d != kD128 || qa.q_gain || !args.out)
        return cudaErrorInvalidValue;
    AttnArgs at = args;
    const cudaError_t me = attention_pool_maps(at);
    if (me != cudaSuccess) return me;
    if (fmt == kFmtInt4) return launch_f<kFmtInt4>(lc, qa, at);
    if (fmt == kFmtInt8) return launch_f<kFmtInt8>(lc, qa, at);
    return cudaErrorInvalidValue;
}

}  // namespace qd
