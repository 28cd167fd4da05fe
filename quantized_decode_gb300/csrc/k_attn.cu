// k_attn.cu - split-K grouped-query decode attention over the paged bf16 KV cache.
//
// Grid (P, Hkv): CTA (p, g) owns KV head g and a contiguous run of pages of
// the T = pos + 1 cached tokens, and serves all G = Hq/Hkv query heads of the
// group from one read of its K/V pages (K and V are read once per KV head,
// not once per query head).  Pages move HBM -> shared memory with cp.async,
// double-buffered.  Per page of 16 tokens:
//   scores:  16 threads per token, each a d/16 slice of q (in registers) . k
//   softmax: online (running max m, running sum l), base-2 exponentials
//   values:  each thread owns 2 dims of the output for every head
// The CTA's unnormalised partial (m, l, o) goes to a scratch slot; the CTA
// that arrives last for KV head g (arrival counter, no waiting) merges the P
// partials with the log-sum-exp weights e^(m_p - M) / sum_p e^(m_p - M) l_p.
#include "common.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kNT = 256;
constexpr float kLog2e = 1.4426950408889634f;

QD_DEV void cp_async16(void *smem, const void *gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
QD_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QD_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

template <int G, int D>
__global__ void __launch_bounds__(kNT) k_attn(AttnArgs a) {
    constexpr int TPT = 16;           // threads per token (score phase)
    constexpr int DPT = D / TPT;      // dims per thread (8 or 4)
    constexpr int NP = D / 2;         // dim pairs
    constexpr int TG = kNT / NP;      // token groups in the value phase (4 or 8)
    constexpr int TPG = 16 / TG;      // tokens per group (4 or 2)
    constexpr int PAGE_ELEMS = kPageTokens * D;
    constexpr int CHUNKS = PAGE_ELEMS * 2 / 16;  // 16-byte chunks per page (256 or 128)

    __shared__ __align__(16) uint16_t ks[2][PAGE_ELEMS];
    __shared__ __align__(16) uint16_t vs[2][PAGE_ELEMS];
    __shared__ __align__(16) float s_sc[16][8];
    __shared__ __align__(16) float s_p[16][8];
    __shared__ float s_alpha[8], s_m[8], s_l[8];
    __shared__ __align__(16) float s_o[TG][G][D];
    __shared__ float s_w[8][256];
    __shared__ int s_last;

    const int p = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
    const int P = gridDim.x;

    pdl_wait();
    const int T = a.T_fixed >= 0 ? a.T_fixed : a.st->pos + 1;
    const int n_pg = (T + kPageTokens - 1) / kPageTokens;
    const int cpp = (n_pg + P - 1) / P;
    const int pg0 = p * cpp;
    const int pg1 = min(n_pg, pg0 + cpp);

    const int tok = tid / TPT, part = tid % TPT;
    const int dp = tid % NP, tg = tid / NP;
    const float qscale = rsqrtf((float)D) * kLog2e;

    float qr[G][DPT];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < DPT; ++e) qr[h][e] = __ldcg(a.q + (size_t)(g * G + h) * D + part * DPT + e) * qscale;

    float2 o[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o[h] = make_float2(0.f, 0.f);
    if (tid < 8) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
    }

    auto issue_page = [&](int pg, int buf) {
        const int phys = __ldg(a.page_table + pg);
        const bool ok = phys >= 0 && phys < a.n_pages;
        const size_t off = ((size_t)(ok ? phys : 0) * a.Hkv + g) * PAGE_ELEMS;
        for (int c = tid; c < CHUNKS; c += kNT) {
            cp_async16(&ks[buf][c * 8], a.k_pool + off + c * 8);
            cp_async16(&vs[buf][c * 8], a.v_pool + off + c * 8);
        }
        if (!ok && tid == 0) atomicCAS(a.err, kErrNone, kErrBadPage);
        cp_async_commit();
    };

    pdl_launch();
    if (pg0 < pg1) issue_page(pg0, 0);
    __syncthreads();
    for (int pg = pg0; pg < pg1; ++pg) {
        const int buf = (pg - pg0) & 1;
        if (pg + 1 < pg1) {
            issue_page(pg + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();

        // ---- scores
        {
            float kf[DPT];
            const uint16_t *kr = &ks[buf][tok * D + part * DPT];
            if constexpr (DPT == 8) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(kr);
                const uint32_t wv[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    kf[2 * e] = __uint_as_float(wv[e] << 16);
                    kf[2 * e + 1] = __uint_as_float(wv[e] & 0xFFFF0000u);
                }
            } else {
                const uint2 raw = *reinterpret_cast<const uint2 *>(kr);
                kf[0] = __uint_as_float(raw.x << 16);
                kf[1] = __uint_as_float(raw.x & 0xFFFF0000u);
                kf[2] = __uint_as_float(raw.y << 16);
                kf[3] = __uint_as_float(raw.y & 0xFFFF0000u);
            }
            float acc[G];
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < DPT; ++e) s = fmaf(qr[h][e], kf[e], s);
                acc[h] = s;
            }
#pragma unroll
            for (int h = 0; h < G; ++h) {
#pragma unroll
                for (int off = TPT / 2; off > 0; off >>= 1) acc[h] += __shfl_xor_sync(0xffffffffu, acc[h], off);
            }
            const bool valid = pg * kPageTokens + tok < T;
#pragma unroll
            for (int h = 0; h < G; ++h)
                if (part == h) s_sc[tok][h] = valid ? acc[h] : -INFINITY;
        }
        __syncthreads();

        // ---- online softmax update: 16 lanes per head; whole warps take part in
        // the shuffles, lanes of heads >= G carry no data.
        if (tid < ((16 * G + 31) / 32) * 32) {
            const int tk = tid & 15, h = tid >> 4;
            const bool act = h < G;
            const float s = act ? s_sc[tk][h] : -INFINITY;
            float pm = s;
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, off));
            const float m_old = act ? s_m[h] : 0.f;
            const float m_new = fmaxf(m_old, pm);
            const float pr = act ? exp2f(s - m_new) : 0.f;
            if (act) s_p[tk][h] = pr;
            float ps = pr;
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
            if (act && tk == 0) {
                const float alpha = exp2f(m_old - m_new);
                s_alpha[h] = alpha;
                s_l[h] = s_l[h] * alpha + ps;
                s_m[h] = m_new;
            }
        }
        __syncthreads();

        // ---- values
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float al = s_alpha[h];
            o[h].x *= al;
            o[h].y *= al;
        }
#pragma unroll
        for (int tt = 0; tt < TPG; ++tt) {
            const int t = tg * TPG + tt;
            if (pg * kPageTokens + t >= T) break;  // slots past the sequence may hold stale rows
            const uint32_t vv = *reinterpret_cast<const uint32_t *>(&vs[buf][t * D + 2 * dp]);
            const float v0 = __uint_as_float(vv << 16), v1 = __uint_as_float(vv & 0xFFFF0000u);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float pr = s_p[t][h];
                o[h].x = fmaf(pr, v0, o[h].x);
                o[h].y = fmaf(pr, v1, o[h].y);
            }
        }
        __syncthreads();
    }

    // ---- this CTA's partial: sum the token groups
#pragma unroll
    for (int h = 0; h < G; ++h) *reinterpret_cast<float2 *>(&s_o[tg][h][2 * dp]) = o[h];
    __syncthreads();
    const size_t slot = (size_t)g * P + p;
    for (int idx = tid; idx < G * D; idx += kNT) {
        const int h = idx / D, dd = idx % D;
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < TG; ++q) s += s_o[q][h][dd];
        a.part_o[slot * G * D + idx] = s;
    }
    if (tid < G) {
        a.part_ml[(slot * G + tid) * 2 + 0] = s_m[tid];
        a.part_ml[(slot * G + tid) * 2 + 1] = s_l[tid];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(a.counter + g, 1) == P - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- combine the P partials of KV head g (P <= 256)
    for (int idx = tid; idx < G * P; idx += kNT) {
        const int h = idx / P, q = idx % P;
        s_w[h][q] = __ldcg(a.part_ml + (((size_t)g * P + q) * G + h) * 2);
    }
    __syncthreads();
    if (tid < G) {
        const int h = tid;
        float M = -INFINITY;
        for (int q = 0; q < P; ++q) M = fmaxf(M, s_w[h][q]);
        float den = 0.f;
        for (int q = 0; q < P; ++q) {
            const float l = __ldcg(a.part_ml + (((size_t)g * P + q) * G + h) * 2 + 1);
            const float w = s_w[h][q] == -INFINITY ? 0.f : exp2f(s_w[h][q] - M);
            s_w[h][q] = w;
            den += w * l;
        }
        s_alpha[h] = 1.f / den;
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kNT) {
        const int h = idx / D;
        float num = 0.f;
        for (int q = 0; q < P; ++q) {
            const float w = s_w[h][q];
            if (w != 0.f) num = fmaf(w, __ldcg(a.part_o + ((size_t)g * P + q) * G * D + idx), num);
        }
        a.out[(size_t)(g * G) * D + idx] = num * s_alpha[h];
    }
    if (tid == 0) a.counter[g] = 0;
}

template <int G>
cudaError_t launch_g(const LaunchCfg &lc, const AttnArgs &a) {
    const dim3 grid(a.P, a.Hkv);
    if (a.d == 128) return launch_k(lc, k_attn<G, 128>, grid, dim3(kNT), 0, a);
    if (a.d == 64) return launch_k(lc, k_attn<G, 64>, grid, dim3(kNT), 0, a);
    return cudaErrorInvalidValue;
}

}  // namespace

int default_splits(int n_sm, int Hkv, int max_pages) {
    int P = (n_sm + Hkv - 1) / Hkv;
    if (P > max_pages) P = max_pages;
    if (P > 256) P = 256;
    return P < 1 ? 1 : P;
}

cudaError_t launch_attention(const LaunchCfg &lc, const AttnArgs &a) {
    if (a.P < 1 || a.P > 256 || a.Hkv < 1 || a.Hq % a.Hkv) return cudaErrorInvalidValue;
    switch (a.Hq / a.Hkv) {
        case 1: return launch_g<1>(lc, a);
        case 2: return launch_g<2>(lc, a);
        case 3: return launch_g<3>(lc, a);
        case 4: return launch_g<4>(lc, a);
        case 5: return launch_g<5>(lc, a);
        case 6: return launch_g<6>(lc, a);
        case 7: return launch_g<7>(lc, a);
        case 8: return launch_g<8>(lc, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qd
