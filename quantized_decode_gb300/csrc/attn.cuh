// attn.cuh - device body of split-K grouped-query decode attention over the
// paged bf16 KV cache, shared by the attention kernel and the fused
// QKV + attention kernel (see k_attn.cu for the algorithm).
#pragma once

#include <cooperative_groups.h>

#include "common.cuh"
#include "gemv.cuh"
#include "ptx.cuh"

namespace qd {

namespace cg = cooperative_groups;

namespace attn {

constexpr int kCS = 8;        // CTAs per cluster (portable size)
constexpr int kCSWide = 16;   // one cluster per KV head (non-portable size)
constexpr int kCSSmall = 4;   // several sequences at once (multi-sequence decode)
constexpr int kWarps = 8;
constexpr int kNT = kWarps * 32;
constexpr int kWRing = 2;     // page slots per warp
constexpr float kLog2e = 1.4426950408889634f;

QD_DEV void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}
QD_DEV void ldsm_x4_t(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(a));
}

// d[0..3] += A(16x16, rows 0-7 from a0/a2, rows 8-15 zero) * B(16x8)
QD_DEV void mma_bf16(float (&d)[2], float &z2, float &z3, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(z2), "+f"(z3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// Split two fp32 values into bf16 hi and lo pairs (x = hi + lo up to 2^-16 |x|).
QD_DEV void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <int D>
constexpr size_t ring_bytes() {
    return (size_t)kWarps * kWRing * 2 * 16 * D * 2;
}
// Dynamic shared memory to request for the ring: its base is rounded up to
// 1024 bytes (the 128-byte swizzle atom of the TMA page boxes).
template <int D>
constexpr size_t ring_alloc_bytes() {
    return ring_bytes<D>() + 1024;
}
QD_DEV uint16_t *align_ring(uint16_t *p) {
    return reinterpret_cast<uint16_t *>(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// A K (or V) page slice in shared memory: 16 rows x D bf16 as D / 64 TMA boxes
// of 16 rows x 128 bytes, each with the 128-byte swizzle (16-byte chunk c of
// row r at chunk c ^ (r & 7) of its 128-byte line), so that the 8 rows an
// ldmatrix reads at one chunk hit distinct banks.  Element offset of (row r,
// 16-byte chunk ch of the D-element row).
QD_DEV int page_off(int r, int ch) { return (ch >> 3) * (16 * 64) + r * 64 + (((ch & 7) ^ (r & 7)) << 3); }

constexpr uint64_t kPageWaitNs = 1000000000ull;  // bound on a page's arrival
// Where a CTA finds its inputs once they exist: the group's G query rows
// (D floats each, RoPE applied) and the appended K and V rows (bf16, D each;
// null when every row is in the pages already).
struct AttnInputs {
    const float *q;
    const uint16_t *k_new, *v_new;
};

// One CTA of split-K decode attention over KV head blockIdx.y (split
// blockIdx.x of gridDim.x, in clusters of CS).  `hook(issue_pages)` waits for
// the producers of the query and of the appended K/V row and returns where
// they are (AttnInputs; QS: in shared memory, else global memory written by an
// earlier kernel).  The CTA's first page copies go out before the hook, or
// (LATE) when the hook calls issue_pages() -- the hook may use the page ring's
// shared memory until then.  smem: ring_bytes<D>() of dynamic shared memory.
// FOLD: the o_proj fold of a.fold is compiled in (the kernel without it has none of its code).
template <int G, int D, int CS, bool QS, bool LATE, class Hook, bool FOLD = false>
QD_DEV void attn_cta(const AttnArgs &a, uint16_t *smem, Hook &&hook) {
    constexpr int CH = D / 8;      // 16-byte chunks per row
    constexpr int PAGE = 16 * D;   // bf16 elements of one K (or V) page slice
    constexpr int NKK = D / 16;    // k-steps of S = Q K^T
    constexpr int NDT = D / 8;     // 8-wide d tiles of O

    __shared__ float s_cm[8], s_cl[8];
    __shared__ __align__(16) float s_co[8][D];
    __shared__ float s_fw[8][32], s_fl[8][32];
    __shared__ float s_st[2][kWarps];
    __shared__ int s_last;
    __shared__ uint64_t s_wbar;  // o_proj fold: the W_o slice has landed
    __shared__ uint64_t s_pbar[kWarps][kWRing];  // page slot arrivals (TMA transaction bytes)

    cg::cluster_group cluster = cg::this_cluster();
    const int g = blockIdx.y, p = blockIdx.x, P = gridDim.x;
    const int rank = (int)cluster.block_rank();
    const int C = P / CS, ci = p / CS;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int gq = lane >> 2, tq = lane & 3;

    // ---- before the wait: only data that is final before the step
    const int T = a.T_fixed >= 0 ? a.T_fixed : a.st->pos + 1;
    const int n_pg = (T + kPageTokens - 1) / kPageTokens;
    const int cpp = (n_pg + P - 1) / P;
    const int pg0 = p * cpp;
    const int pg1 = min(n_pg, pg0 + cpp);
    const int n = pg1 > pg0 ? pg1 - pg0 : 0;
    const int nw = n > warp ? (n - 1 - warp) / kWarps + 1 : 0;  // this warp's pages
    uint16_t *wring = smem + (size_t)warp * kWRing * 2 * PAGE;  // 1024-byte aligned: smem is, slots are 8 KB
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < kWRing; ++j) ptx::mbar_init(&s_pbar[warp][j], 1);
        ptx::mbar_fence_init();
    }
    __syncwarp();

    // page i of this warp into slot i % kWRing: lane 0 issues the K and V boxes
    // (TMA), the slot's barrier counts their bytes
    auto issue = [&](int i) {
        if (lane != 0) return;
        const int pg = pg0 + warp + i * kWarps;
        const int phys = __ldg(a.page_table + pg);
        const bool ok = phys >= 0 && phys < a.n_pages;
        if (!ok) atomicCAS(a.err, kErrNone, kErrBadPage);
        const int row = ((ok ? phys : 0) * a.Hkv + g) * kPageTokens;
        uint16_t *ks = wring + (i % kWRing) * 2 * PAGE, *vs = ks + PAGE;
        uint64_t *bar = &s_pbar[warp][i % kWRing];
        ptx::fence_proxy_async_smem();  // the warp's earlier accesses of the slot come before the copy's writes
        ptx::mbar_expect_tx(bar, (uint32_t)(2 * PAGE * 2));
#pragma unroll
        for (int b = 0; b < D / 64; ++b) {
            ptx::tma_load_2d(ks + b * 16 * 64, &a.k_map, b * 64, row, bar);
            ptx::tma_load_2d(vs + b * 16 * 64, &a.v_map, b * 64, row, bar);
        }
    };
    auto issue_pages = [&]() {
#pragma unroll
        for (int i = 0; i < kWRing; ++i)
            if (i < nw) issue(i);
    };
    if (!LATE) issue_pages();

    const AttnInputs in = hook(issue_pages);

    // ---- query fragments: rows = heads (gq < G), k = d; hi and lo bf16 parts
    uint32_t qh[NKK][2], ql[NKK][2];
#pragma unroll
    for (int kk = 0; kk < NKK; ++kk)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int d0 = kk * 16 + hf * 8 + 2 * tq;
            float q0 = 0.f, q1 = 0.f;
            if (gq < G) {
                const float2 *qp = reinterpret_cast<const float2 *>(in.q + (size_t)gq * D + d0);
                const float2 qv = QS ? *qp : __ldcg(qp);
                q0 = qv.x;
                q1 = qv.y;
            }
            split2(q0, q1, qh[kk][hf], ql[kk][hf]);
        }
    const float sscale = rsqrtf((float)D) * kLog2e;
    // the appended row (position T-1) is taken from kv_new when given
    const int last_pg = n_pg - 1, new_row = (T - 1) % kPageTokens;
    const bool patch = in.k_new != nullptr;

    float m = -INFINITY, l = 0.f;
    float o[NDT][2];
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) o[dt][0] = o[dt][1] = 0.f;
    float z2 = 0.f, z3 = 0.f;  // rows 8-15 of the products (always zero)

    int stop = nw;  // pages consumed; < nw only if a page's arrival wait ran out
    for (int i = 0; i < nw; ++i) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&s_pbar[warp][i % kWRing], (i / kWRing) & 1u, kPageWaitNs))) {
            if (lane == 0) atomicCAS(a.err, kErrNone, kErrTimeout);
            stop = i;
            break;
        }
        const int pg = pg0 + warp + i * kWarps;
        uint16_t *ks = wring + (i % kWRing) * 2 * PAGE, *vs = ks + PAGE;
        if (pg == last_pg) {
            const int valid = T - pg * kPageTokens;  // rows [valid, 16) lie past the sequence
            for (int c = lane; c < (16 - valid) * CH; c += 32) {
                const int r = valid + c / CH, ch = c % CH;
                *reinterpret_cast<uint4 *>(vs + page_off(r, ch)) = make_uint4(0, 0, 0, 0);
            }
            if (patch && lane < CH) {
                const int sw = page_off(new_row, lane);
                const uint4 *kn = reinterpret_cast<const uint4 *>(in.k_new) + lane;
                const uint4 *vn = reinterpret_cast<const uint4 *>(in.v_new) + lane;
                *reinterpret_cast<uint4 *>(ks + sw) = QS ? *kn : __ldcg(kn);
                *reinterpret_cast<uint4 *>(vs + sw) = QS ? *vn : __ldcg(vn);
            }
            __syncwarp();
        }

        // ---- S = Q K^T for the 16 tokens of the page (two n-tiles of 8)
        float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < NKK; ++kk) {
            const int tok = (lane & 7) + ((lane >> 4) << 3);
            const int ch = kk * 2 + ((lane >> 3) & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(ks + page_off(tok, ch), b0, b1, b2, b3);
            mma_bf16(s0, z2, z3, qh[kk][0], qh[kk][1], b0, b1);
            mma_bf16(s0, z2, z3, ql[kk][0], ql[kk][1], b0, b1);
            mma_bf16(s1, z2, z3, qh[kk][0], qh[kk][1], b2, b3);
            mma_bf16(s1, z2, z3, ql[kk][0], ql[kk][1], b2, b3);
        }
        // thread holds head gq, tokens 2tq, 2tq+1 (s0) and 8+2tq, 9+2tq (s1)
        const int base = pg * kPageTokens;
        float v0 = base + 2 * tq < T ? s0[0] * sscale : -INFINITY;
        float v1 = base + 2 * tq + 1 < T ? s0[1] * sscale : -INFINITY;
        float v2 = base + 8 + 2 * tq < T ? s1[0] * sscale : -INFINITY;
        float v3 = base + 9 + 2 * tq < T ? s1[1] * sscale : -INFINITY;
        float mx = fmaxf(fmaxf(v0, v1), fmaxf(v2, v3));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m, mx);  // finite: every processed page holds a valid token
        const float alpha = exp2f(m - m_new);
        const float p0 = exp2f(v0 - m_new), p1 = exp2f(v1 - m_new);
        const float p2 = exp2f(v2 - m_new), p3 = exp2f(v3 - m_new);
        float ps = (p0 + p1) + (p2 + p3);
        ps += __shfl_xor_sync(0xffffffffu, ps, 1);
        ps += __shfl_xor_sync(0xffffffffu, ps, 2);
        l = l * alpha + ps;
        m = m_new;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt) {
            o[dt][0] *= alpha;
            o[dt][1] *= alpha;
        }
        uint32_t ph0, pl0, ph2, pl2;
        split2(p0, p1, ph0, pl0);
        split2(p2, p3, ph2, pl2);

        // ---- O += P V (16 tiles of 8 dims, two per ldmatrix)
#pragma unroll
        for (int dp = 0; dp < NDT / 2; ++dp) {
            const int mi = lane >> 3, r = lane & 7;
            const int tok = r + (mi & 1) * 8;
            const int ch = dp * 2 + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vs + page_off(tok, ch), b0, b1, b2, b3);
            mma_bf16(o[2 * dp], z2, z3, ph0, ph2, b0, b1);
            mma_bf16(o[2 * dp], z2, z3, pl0, pl2, b0, b1);
            mma_bf16(o[2 * dp + 1], z2, z3, ph0, ph2, b2, b3);
            mma_bf16(o[2 * dp + 1], z2, z3, pl0, pl2, b2, b3);
        }
        __syncwarp();
        if (i + kWRing < nw) issue(i + kWRing);
    }
    // after a wait ran out: the pages still in flight land before the slots are reused
    for (int i = stop; i < nw && i < stop + kWRing; ++i)
        ptx::mbar_wait(&s_pbar[warp][i % kWRing], (i / kWRing) & 1u, kPageWaitNs);
    __syncthreads();

    // ---- merge the 8 warps of the CTA (the ring's shared memory is free now)
    float *wm = reinterpret_cast<float *>(smem);  // [warps][8]
    float *wl = wm + kWarps * 8;                   // [warps][8]
    float *wo = wl + kWarps * 8;                   // [warps][8][D]
    if (tq == 0) {
        wm[warp * 8 + gq] = nw > 0 ? m : -INFINITY;
        wl[warp * 8 + gq] = nw > 0 ? l : 0.f;
    }
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) {
        wo[(warp * 8 + gq) * D + dt * 8 + 2 * tq] = o[dt][0];
        wo[(warp * 8 + gq) * D + dt * 8 + 2 * tq + 1] = o[dt][1];
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kNT) {
        const int h = idx / D, dim = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w * 8 + h]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = exp2f(wm[w * 8 + h] - M);
                num = fmaf(f, wo[(w * 8 + h) * D + dim], num);
                den = fmaf(f, wl[w * 8 + h], den);
            }
        }
        s_co[h][dim] = num;
        if (dim == 0) {
            s_cm[h] = M;
            s_cl[h] = den;
        }
    }
    const bool fold = FOLD && C == 1 && a.out != nullptr && a.fold != nullptr;
    const int fold_rows = fold ? a.fold->hidden / CS : 0;
    constexpr int kFoldRowBytes = G * D / 2;  // one W_o row's INT4 codes for this KV head's columns
    if constexpr (FOLD) {
        if (fold) ptx::fence_proxy_async_smem();  // the warp merge's writes come before the copies' writes
    }
    cluster.sync();
    // o_proj fold: this CTA's rows of W_o (its KV head's columns) into the free page ring,
    // landing while the cluster merges
    // ring layout of the fold: W_o rows | outputs fp16 | outputs fp32 | group scales | this CTA's
    // merged outputs (read by the other CTAs of the cluster; the same offset in every CTA)
    constexpr int kFoldGroups = G * D / kGroup;  // scale groups of a row in this KV head's columns
    uint16_t *fold_sc = reinterpret_cast<uint16_t *>(reinterpret_cast<char *>(smem) + (size_t)fold_rows * kFoldRowBytes +
                                                     (size_t)G * D * 6);
    float *s_vec = reinterpret_cast<float *>(
        reinterpret_cast<char *>(smem) +
        (((size_t)fold_rows * kFoldRowBytes + (size_t)G * D * 6 + (size_t)fold_rows * kFoldGroups * 2 + 15) & ~(size_t)15));
    if constexpr (FOLD) {
    if (fold && tid == 0) {
        ptx::mbar_init(&s_wbar, 1);
        ptx::mbar_fence_init();
        ptx::mbar_expect_tx(&s_wbar, (uint32_t)(fold_rows * kFoldRowBytes));
        ptx::tma_load_2d(smem, &a.fold->wo_map, g * (kFoldRowBytes / 4), rank * fold_rows, &s_wbar);
    }
    if constexpr (kFoldGroups > 0) {
        if (fold) {  // this CTA's rows' scales (static weights), read once, in flight during the merge
            const int groups = a.Hq * D / kGroup, r0 = rank * fold_rows;
            for (int u = tid; u < fold_rows * kFoldGroups; u += kNT)
                fold_sc[u] = __ldg(a.fold->so + (size_t)(r0 + u / kFoldGroups) * groups + g * kFoldGroups + u % kFoldGroups);
        }
    }
    }

    // ---- merge the CS CTAs of the cluster through distributed shared memory;
    // rank r merges an equal slice of the G*D outputs into the cluster's partial,
    // or, with one cluster per KV head, into the final output
    const bool direct = C == 1 && a.out != nullptr;
    float st_ss = 0.f, st_mx = 0.f;
    {
        const int per = (G * D + CS - 1) / CS;
        const int lo = rank * per, hi = min(G * D, lo + per);
        for (int idx = lo + tid; idx < hi; idx += kNT) {
            const int h = idx / D, dim = idx % D;
            float M = -INFINITY;
#pragma unroll
            for (int q = 0; q < CS; ++q) M = fmaxf(M, cluster.map_shared_rank(s_cm, q)[h]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int q = 0; q < CS; ++q) {
                    const float f = exp2f(cluster.map_shared_rank(s_cm, q)[h] - M);
                    num = fmaf(f, cluster.map_shared_rank(&s_co[0][0], q)[h * D + dim], num);
                    den = fmaf(f, cluster.map_shared_rank(s_cl, q)[h], den);
                }
            }
            if (direct) {  // den > 0: the cluster holds every token
                const float v = num * (1.f / den);
                if constexpr (FOLD) {
                    if (fold) {
                        s_vec[idx - lo] = v;
                        continue;
                    }
                }
                a.out[(size_t)(g * G) * D + idx] = v;
                st_ss += v * v;
                st_mx = fmaxf(st_mx, fabsf(v));
                continue;
            }
            const size_t slot = (size_t)g * C + ci;
            a.part_o[(slot * G + h) * D + dim] = num;
            if (dim == 0) {
                a.part_ml[(slot * G + h) * 2] = M;
                a.part_ml[(slot * G + h) * 2 + 1] = den;
            }
        }
    }
    if constexpr (FOLD) {
    if (fold) {
        // every CTA's merged slice is in its s_vec; the merge's reads of s_co are done
        cluster.sync();
        const int per = (G * D + CS - 1) / CS;
        // the cluster's G*D outputs as fp16 scaled by 2^-e (|x| <= 1) after the W_o slice
        __half *xh = reinterpret_cast<__half *>(reinterpret_cast<char *>(smem) + (size_t)fold_rows * kFoldRowBytes);
        float *xf = reinterpret_cast<float *>(xh + G * D);  // fp32 copy of the gathered vector
        float mx = 0.f;
        for (int idx = tid; idx < G * D; idx += kNT) {
            const float v = cluster.map_shared_rank(s_vec, (unsigned)(idx / per))[idx % per];
            xf[idx] = v;
            mx = fmaxf(mx, fabsf(v));
        }
        // this CTA's reads of its peers' shared memory are done; leave only after all peers' are
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        mx = warp_max(mx);
        if (lane == 0) s_st[1][warp] = mx;
        __syncthreads();
        float gmx = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) gmx = fmaxf(gmx, s_st[1][w]);
        int e = 0;
        if (gmx > 0.f) frexpf(gmx, &e);  // gmx < 2^e
        const float down = ldexpf(1.f, -e), up = ldexpf(1.f, e);
        for (int idx = tid; idx < G * D; idx += kNT) xh[idx] = __float2half_rn(xf[idx] * down);
        __syncthreads();
        const bool landed = ptx::mbar_wait(&s_wbar, 0, kPageWaitNs);
        if (!landed && tid == 0) atomicCAS(a.err, kErrNone, kErrTimeout);
        // warp w: rows [w R, w R + R) of the CTA's slice; lane l < G*D/32: codes 32 l .. 32 l + 31
        constexpr int kUnits = G * D / 32;
        const int R = fold_rows / kWarps, r0 = rank * fold_rows;
        const uint4 *wq = reinterpret_cast<const uint4 *>(smem);
        const uint4 *xq = reinterpret_cast<const uint4 *>(xh);
        const int ul = lane < kUnits ? lane : 0;
        const uint4 x[4] = {xq[4 * ul], xq[4 * ul + 1], xq[4 * ul + 2], xq[4 * ul + 3]};
        // four rows at a time: independent dot products and reductions in flight together
        for (int i0 = warp * R; landed && i0 < warp * R + R; i0 += 4) {
            float v[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int i = i0 + k;
                v[k] = 0.f;
                if (i < warp * R + R && lane < kUnits)
                    v[k] = int4_unit_dot(wq[(size_t)i * kUnits + lane], x) *
                           bf16_bits_to_float(fold_sc[i * kFoldGroups + lane / 4]);
            }
#pragma unroll
            for (int o2 = 16; o2 > 0; o2 >>= 1)
#pragma unroll
                for (int k = 0; k < 4; ++k) v[k] += __shfl_xor_sync(0xffffffffu, v[k], o2);
            if (lane == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    if (i0 + k < warp * R + R)
                        atomicAdd(reinterpret_cast<unsigned long long *>(a.fold->out + r0 + i0 + k),
                                  (unsigned long long)delta_to_fixed(v[k] * up));
            }
        }
        if (!landed) ptx::mbar_wait(&s_wbar, 0, kPageWaitNs);  // copies still in flight land first
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        return;
    }
    }
    if (direct) {
        // this CTA's reads of its peers' shared memory are done: arrive now and
        // wait only before leaving (no CTA leaves while a peer may still read its
        // shared memory), so the statistics overlap the barrier
        asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
        if (a.stats_out) {  // one (ss, mx) slot per CTA: g * CS + rank
            st_ss = warp_sum(st_ss);
            st_mx = warp_max(st_mx);
            if (lane == 0) {
                s_st[0][warp] = st_ss;
                s_st[1][warp] = st_mx;
            }
            __syncthreads();
            if (tid == 0) {
                float a0 = 0.f, b0 = 0.f;
                for (int w = 0; w < kWarps; ++w) {
                    a0 += s_st[0][w];
                    b0 = fmaxf(b0, s_st[1][w]);
                }
                a.stats_out[2 * (g * CS + rank)] = a0;
                a.stats_out[2 * (g * CS + rank) + 1] = b0;
            }
        }
        asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
        return;
    }
    __threadfence();
    cluster.sync();  // no CTA leaves while a peer may still read its shared memory
    if (rank != 0) return;
    if (tid == 0) s_last = atomicAdd(a.counter + g, 1) == C - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    // ---- last cluster of KV head g: merge the C cluster partials (C <= 32)
    if (tid < G * C) {
        const int h = tid / C, c = tid % C;
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(a.part_ml) + ((size_t)g * C + c) * G + h);
        s_fw[h][c] = ml.x;
        s_fl[h][c] = ml.y;
    }
    __syncthreads();
    if (tid < G) {
        float M = -INFINITY;
        for (int c = 0; c < C; ++c) M = fmaxf(M, s_fw[tid][c]);
        float den = 0.f;
        for (int c = 0; c < C; ++c) {
            const float f = s_fw[tid][c] == -INFINITY ? 0.f : exp2f(s_fw[tid][c] - M);
            den = fmaf(f, s_fl[tid][c], den);
            s_fw[tid][c] = f;
        }
        s_cl[tid] = 1.f / den;
    }
    __syncthreads();
    float mx = 0.f, ss = 0.f;
    // every output of the thread at once, the cluster partials four at a time:
    // the L2 reads of a batch are in flight together
    constexpr int kPer = (G * D + kNT - 1) / kNT;
    float num[kPer];
#pragma unroll
    for (int r = 0; r < kPer; ++r) num[r] = 0.f;
#pragma unroll 4
    for (int c = 0; c < C; ++c) {
#pragma unroll
        for (int r = 0; r < kPer; ++r) {
            const int idx = tid + r * kNT;
            if (idx < G * D) {
                const int h = idx / D, dim = idx % D;
                num[r] = fmaf(s_fw[h][c], __ldcg(a.part_o + (((size_t)g * C + c) * G + h) * D + dim), num[r]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < kPer; ++r) {
        const int idx = tid + r * kNT;
        if (idx < G * D) {
            const float v = num[r] * s_cl[idx / D];
            a.out[(size_t)(g * G) * D + idx] = v;
            mx = fmaxf(mx, fabsf(v));
            ss += v * v;
        }
    }
    if (a.stats_out) {
        ss = warp_sum(ss);
        mx = warp_max(mx);
        if (lane == 0) {
            s_co[0][warp] = ss;
            s_co[1][warp] = mx;
        }
        __syncthreads();
        if (tid == 0) {
            float a0 = 0.f, b0 = 0.f;
            for (int w = 0; w < kWarps; ++w) {
                a0 += s_co[0][w];
                b0 = fmaxf(b0, s_co[1][w]);
            }
            a.stats_out[2 * g] = a0;
            a.stats_out[2 * g + 1] = b0;
        }
    }
    if (tid == 0) a.counter[g] = 0;
}

}  // namespace attn

}  // namespace qd
