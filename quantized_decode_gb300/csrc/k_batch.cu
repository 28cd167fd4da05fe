// k_batch.cu - kernels of the multi-sequence decode step (batch.cu): up to 8
// sequences decode together, each through its own page table, and every weight
// is read once per step for all of them ("Systems Foundations for LLMs",
// PagedAttention: per-sequence block tables over one shared pool of 16-token
// blocks).
//
// The linear layers become skinny GEMMs, Y[b][n] = sum_k W[n][k] X[b][k] for
// b < B <= 8, run on the tensor cores with mma.sync m16n8k16 (bf16 operands,
// fp32 accumulation): A = 16 weight rows, their INT4 / INT8 codes turned into
// exact bf16 integers in registers (bf16 weights as they are); B = the 8
// sequences' activations, staged in shared memory as bf16
// after the RMSNorm; the column n of the mma is the sequence.  INT4 group
// scales are applied to the fp32 partial sum of each 128-code group, INT8 row
// scales at the end.  Each warp streams its rows' 64-byte blocks through a
// cp.async ring in shared memory, kRD - 1 blocks ahead of the arithmetic.
#include <cuda_bf16.h>

#include "common.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kNW = 8;        // warps per CTA
constexpr int kKC = 12288;    // K values staged in shared memory at a time (192 KB for 8 sequences)
constexpr int kTPW = 8;       // row tiles per warp at most (fp32 accumulators)
constexpr int kRD = 12;       // weight ring stages per warp (64-byte blocks of its two rows, cp.async)
constexpr int kRingWarpBytes = kRD * 2 * 32 * (16 + 4);  // codes + INT4 scale words, per warp
constexpr int kRedEntries = kNW * kTPW * 4 * 32 * 4 / 16;  // 16-byte entries of the K-part sums
constexpr int kNormK = 4096;  // RMSNorm'd inputs: K at most this

QD_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                     uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// bf16x2 (x - 136, y - 136): exact for the integers 128 .. 143 the INT4 unpack forms.
QD_DEV uint32_t bf2_minus136(uint32_t v) {
    __nv_bfloat162 a = *reinterpret_cast<__nv_bfloat162 *>(&v);
    const __nv_bfloat162 k = __floats2bfloat162_rn(136.f, 136.f);
    a = __hsub2(a, k);
    return *reinterpret_cast<uint32_t *>(&a);
}

// INT4 ValueShuffle word -> the bf16 pairs (c0,c1), (c2,c3), (c4,c5), (c6,c7).
// A pair's nibbles sit at bits (4j, 16 + 4j); nibble ^ 8 = c + 8 under the bf16
// exponent of 128 (0x4300) is 136 + c, and subtracting 136 is exact.
QD_DEV void int4_word_bf16(uint32_t w, uint32_t (&p)[4]) {
    p[0] = bf2_minus136(lop3_and_xor(w, 0x000F000Fu, 0x43084308u));
    p[1] = bf2_minus136(lop3_and_xor(w >> 4, 0x000F000Fu, 0x43084308u));
    p[2] = bf2_minus136(lop3_and_xor(w >> 8, 0x000F000Fu, 0x43084308u));
    p[3] = bf2_minus136(lop3_and_xor(w >> 12, 0x000F000Fu, 0x43084308u));
}

// INT8 word (natural byte order) -> bf16 pairs (b0,b1), (b2,b3): each byte goes
// under the fp32 exponent of 2^23 ((b ^ 0x80) = c + 128), 2^23 + 128 is
// subtracted exactly and the pair is rounded to bf16 (exact: |c| <= 127).
QD_DEV void int8_word_bf16(uint32_t w, uint32_t (&p)[2]) {
    const uint32_t t = w ^ 0x80808080u;
    const float k = 8388736.f;  // 2^23 + 128
    const float c0 = __uint_as_float(prmt(t, 0x4B000000u, 0x7650u)) - k;
    const float c1 = __uint_as_float(prmt(t, 0x4B000000u, 0x7651u)) - k;
    const float c2 = __uint_as_float(prmt(t, 0x4B000000u, 0x7652u)) - k;
    const float c3 = __uint_as_float(prmt(t, 0x4B000000u, 0x7653u)) - k;
    __nv_bfloat162 a = __floats2bfloat162_rn(c0, c1), b = __floats2bfloat162_rn(c2, c3);
    p[0] = *reinterpret_cast<uint32_t *>(&a);
    p[1] = *reinterpret_cast<uint32_t *>(&b);
}

// Codes of one 16-byte lane chunk per 64-byte row block.
template <int FMT>
constexpr int codes_per_lane() { return FMT == kFmtInt4 ? 32 : (FMT == kFmtInt8 ? 16 : 8); }

// Staged activations: k-chunk c (8 values) of sequence b at 16-byte entry
// c * 8 + (b ^ ((c >> 2) & 7)) (the swizzle spreads a warp's reads over the banks).
QD_DEV int act_entry(int c, int b) { return c * 8 + (b ^ ((c >> 2) & 7)); }

template <int FMT>
__global__ void __launch_bounds__(kNW * 32, 1) k_bgemv(BGemvArgs a) {
    constexpr int CPL = codes_per_lane<FMT>();
    constexpr int NM = CPL / 4;            // mma per 64-byte block
    constexpr int BLK = 4 * CPL;           // K values per 64-byte row block
    extern __shared__ uint4 sx[];          // [kKC / 8][8] 16-byte entries of bf16
    __shared__ float s_inv[8];
    __shared__ float red[kNW][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int tiles = a.mode == 2 ? a.N / 8 : a.N / 16;
    // ks warps share a tile, each over its own part of K (their sums meet in
    // shared memory at the end); the CTA holds kNW / ks tile slots
    const int ks = a.ks, kp = warp % ks, tslots = kNW / ks;
    const int gw = blockIdx.x * tslots + warp / ks, nwarps = gridDim.x * tslots;
    const int B = a.B;
    // shared memory: the staging area for min(K part, kKC) values of 8 sequences (it also
    // holds the K-part sums at the end), then each warp's weight ring
    int stage_entries = (a.K + (int)gridDim.y - 1) / (int)gridDim.y + 128;
    if (stage_entries > kKC) stage_entries = kKC;
    if (stage_entries < kRedEntries) stage_entries = kRedEntries;
    char *ring_base = reinterpret_cast<char *>(sx + stage_entries) + (size_t)warp * kRingWarpBytes;
    uint4 *rc = reinterpret_cast<uint4 *>(ring_base);                    // [kRD][2 rows][32 lanes]
    uint32_t *rs = reinterpret_cast<uint32_t *>(ring_base + kRD * 2 * 32 * 16);  // [kRD][2][32]

    float acc[kTPW][4];
#pragma unroll
    for (int i = 0; i < kTPW; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    // the row pair (g, g + 8) of tile ti: pointers into the weight rows and scales
    auto row_ptrs = [&](int ti, const uint4 *&r0, const uint4 *&r1, const void *&s0, const void *&s1, int &rr0,
                        int &rr1) {
        const size_t rb = FMT == kFmtInt4 ? (size_t)a.K / 2 : (FMT == kFmtInt8 ? (size_t)a.K : (size_t)a.K * 2);
        if (a.mode == 2) {  // 8 gate rows then the same 8 up rows
            const int f = ti * 8 + g;
            r0 = reinterpret_cast<const uint4 *>((const char *)a.w[0] + (size_t)f * rb);
            r1 = reinterpret_cast<const uint4 *>((const char *)a.w2 + (size_t)f * rb);
            s0 = a.s[0];
            s1 = a.s2;
            rr0 = rr1 = f;
            return;
        }
        int r = ti * 16 + g, seg = 0;
        while (seg + 1 < a.n_seg && r >= a.seg_rows[seg]) r -= a.seg_rows[seg++];
        r0 = reinterpret_cast<const uint4 *>((const char *)a.w[seg] + (size_t)r * rb);
        r1 = reinterpret_cast<const uint4 *>((const char *)a.w[seg] + (size_t)(r + 8) * rb);
        s0 = s1 = a.s[seg];
        rr0 = r;
        rr1 = r + 8;
    };

    // grid.y parts of K (large-K projections): this CTA's range of 64-byte blocks
    const int nb_all = a.K / BLK;
    const int kbeg = (int)((long long)nb_all * blockIdx.y / gridDim.y) * BLK;
    const int kend = (int)((long long)nb_all * (blockIdx.y + 1) / gridDim.y) * BLK;

    // Weight stream of a chunk of K: stage f (tile f / nblk, block f % nblk) holds lane t's
    // 16 bytes of the tile's two rows (and, INT4, the word holding each row's group scale)
    // in ring slot f % kRD; kRD - 1 stages are in flight while one is multiplied.
    // issue cursor: tile li, block lb, ring slot ls; the tile's row pointers are found once
    int kb0 = 0, nblk = 0, nt = 0, F = 0, ub0 = 0;
    int li = 0, lb = 0, ls = 0;
    const uint4 *lr0 = nullptr, *lr1 = nullptr;
    const uint32_t *lsc0 = nullptr, *lsc1 = nullptr;
    auto tile_rows = [&](int i) {
        const void *s0, *s1;
        int rr0, rr1;
        row_ptrs(gw + i * nwarps, lr0, lr1, s0, s1, rr0, rr1);
        lr0 += (size_t)ub0 * 4 + t;
        lr1 += (size_t)ub0 * 4 + t;
        if constexpr (FMT == kFmtInt4) {  // scale words: G even (K % 256 == 0), a block's parity picks the half
            const size_t G = (size_t)a.K / kGroup;
            lsc0 = static_cast<const uint32_t *>(s0) + (((size_t)rr0 * G + ub0) >> 1);
            lsc1 = static_cast<const uint32_t *>(s1) + (((size_t)rr1 * G + ub0) >> 1);
        }
    };
    auto issue = [&]() {
        cp_async16(rc + (ls * 2 + 0) * 32 + lane, lr0 + (size_t)lb * 4);
        cp_async16(rc + (ls * 2 + 1) * 32 + lane, lr1 + (size_t)lb * 4);
        if constexpr (FMT == kFmtInt4) {
            const int hw = ((ub0 & 1) + lb) >> 1;  // scale word of block ub0 + lb, from the tile's first
            cp_async4(rs + (ls * 2 + 0) * 32 + lane, lsc0 + hw);
            cp_async4(rs + (ls * 2 + 1) * 32 + lane, lsc1 + hw);
        }
        if (++ls == kRD) ls = 0;
        if (++lb == nblk) {
            lb = 0;
            if (++li < nt) tile_rows(li);
        }
    };
    // the chunk [k0, k0 + kc): this warp's blocks and tiles, and its first kRD - 1 stages
    auto start_chunk = [&](int k0, int kc) {
        const int nblk_all = kc / BLK;
        kb0 = nblk_all * kp / ks;
        const int kb1 = nblk_all * (kp + 1) / ks;  // this warp's blocks of the chunk
        nblk = kb1 - kb0;
        nt = 0;
        while (nt < kTPW && gw + nt * nwarps < tiles) ++nt;
        F = nblk > 0 ? nt * nblk : 0;
        ub0 = k0 / BLK + kb0;  // first block of this warp's part in the row (64-byte units)
        li = lb = ls = 0;
        if (F > 0) tile_rows(0);
        for (int f = 0; f < kRD - 1; ++f) {
            if (f < F) issue();
            cp_async_commit();
        }
    };
    // the first chunk's weights go out before the dependency wait: nothing an earlier
    // kernel writes is read by them, and the ring lies outside the staging area
    start_chunk(kbeg, kend - kbeg < kKC ? kend - kbeg : kKC);

    // programmatic dependent launch: everything below reads or writes activations
    pdl_wait();
    pdl_launch();

    // ---- with an RMSNorm (K <= kNormK): the sums of squares of the B input rows (one pass
    // over them in L2); the staging below reads them again and normalizes
    if (threadIdx.x < 8) s_inv[threadIdx.x] = 1.f;
    if (a.gamma) {
        float ss[8];
#pragma unroll
        for (int b = 0; b < 8; ++b) ss[b] = 0.f;
        constexpr int kB = 4;  // float4 loads per sequence in flight per thread
        for (int k = threadIdx.x * 4; k < a.K; k += blockDim.x * 4 * kB) {
            float4 v[8][kB];
#pragma unroll
            for (int b = 0; b < 8; ++b)
#pragma unroll
                for (int j = 0; j < kB; ++j) {
                    const int kk = k + j * blockDim.x * 4;
                    v[b][j] = b < B && kk < a.K ? __ldcg(reinterpret_cast<const float4 *>(a.x + (size_t)b * a.ldx + kk))
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
            for (int b = 0; b < 8; ++b)
#pragma unroll
                for (int j = 0; j < kB; ++j)
                    ss[b] += v[b][j].x * v[b][j].x + v[b][j].y * v[b][j].y + v[b][j].z * v[b][j].z +
                             v[b][j].w * v[b][j].w;
        }
#pragma unroll
        for (int b = 0; b < 8; ++b) {
            const float v = warp_sum(ss[b]);
            if (lane == 0) red[warp][b] = v;
        }
        __syncthreads();
        if (threadIdx.x < 8) {
            float v = 0.f;
            for (int w = 0; w < kNW; ++w) v += red[w][threadIdx.x];
            s_inv[threadIdx.x] = rsqrtf(v / (float)a.K + a.eps);
        }
    }
    __syncthreads();

#pragma unroll 1
    for (int k0 = kbeg; k0 < kend; k0 += kKC) {
        const int kc = kend - k0 < kKC ? kend - k0 : kKC;
        if (k0 != kbeg) start_chunk(k0, kc);  // the previous chunk's ring is drained
        // ---- stage X[b][k0 .. k0 + kc) as bf16 (normalized), zeros for b >= B, several
        // entries' loads in flight per thread
        __syncthreads();
        constexpr int kE = 4;
        for (int e0 = threadIdx.x; e0 < (kc / 8) * 8; e0 += blockDim.x * kE) {
            float4 v0[kE], v1[kE];
#pragma unroll
            for (int j = 0; j < kE; ++j) {
                const int e = e0 + j * blockDim.x, c = e >> 3, b = e & 7;
                v0[j] = v1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e < (kc / 8) * 8 && b < B) {
                    const float *src = a.x + (size_t)b * a.ldx + k0 + c * 8;
                    v0[j] = __ldcg(reinterpret_cast<const float4 *>(src));
                    v1[j] = __ldcg(reinterpret_cast<const float4 *>(src + 4));
                }
            }
#pragma unroll
            for (int j = 0; j < kE; ++j) {
            const int e = e0 + j * blockDim.x, c = e >> 3, b = e & 7;
            if (e >= (kc / 8) * 8) break;
            uint4 out = make_uint4(0u, 0u, 0u, 0u);
            if (b < B) {
                float f[8] = {v0[j].x, v0[j].y, v0[j].z, v0[j].w, v1[j].x, v1[j].y, v1[j].z, v1[j].w};
                const float inv = s_inv[b];
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float x0 = f[2 * i] * inv, x1 = f[2 * i + 1] * inv;
                    if (a.gamma) {
                        const uint32_t gg = __ldg(reinterpret_cast<const uint32_t *>(a.gamma + k0 + c * 8) + i);
                        x0 *= __uint_as_float(gg << 16);
                        x1 *= __uint_as_float(gg & 0xFFFF0000u);
                    }
                    __nv_bfloat162 h2 = __floats2bfloat162_rn(x0, x1);
                    o[i] = *reinterpret_cast<uint32_t *>(&h2);
                }
                out = make_uint4(o[0], o[1], o[2], o[3]);
            }
            sx[act_entry(c, b)] = out;
            }
        }
        __syncthreads();

        float cur[4] = {0.f, 0.f, 0.f, 0.f};
        int i = 0, bk = 0, slot = 0;  // compute cursor
#pragma unroll 1
        for (int f = 0; f < F; ++f) {
            if (f + kRD - 1 < F) issue();
            cp_async_commit();
            cp_async_wait<kRD - 1>();
            const int cbase = ((kb0 + bk) * BLK + t * CPL) / 8;  // staged k-chunk of this lane's codes
            // A pairs of the two rows
            uint32_t pa[2][CPL / 2];
            const uint4 wv[2] = {rc[(slot * 2 + 0) * 32 + lane], rc[(slot * 2 + 1) * 32 + lane]};
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const uint32_t ww[4] = {wv[r].x, wv[r].y, wv[r].z, wv[r].w};
                if constexpr (FMT == kFmtInt4) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t p[4];
                        int4_word_bf16(ww[j], p);
#pragma unroll
                        for (int z = 0; z < 4; ++z) pa[r][4 * j + z] = p[z];
                    }
                } else if constexpr (FMT == kFmtInt8) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t p[2];
                        int8_word_bf16(ww[j], p);
                        pa[r][2 * j] = p[0];
                        pa[r][2 * j + 1] = p[1];
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) pa[r][j] = ww[j];
                }
            }
            // two accumulator chains (even and odd k-steps) halve the mma dependency chain
            float d[4] = {0.f, 0.f, 0.f, 0.f}, e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int m = 0; m < NM; ++m) {
                // B: this lane's sequence g, k values t*CPL + 4m .. + 3 of the block
                const uint4 xb = sx[act_entry(cbase + (4 * m) / 8, g)];
                const uint32_t b0 = (m & 1) ? xb.z : xb.x, b1 = (m & 1) ? xb.w : xb.y;
                if (m & 1) mma_bf16(e, pa[0][2 * m], pa[1][2 * m], pa[0][2 * m + 1], pa[1][2 * m + 1], b0, b1);
                else mma_bf16(d, pa[0][2 * m], pa[1][2 * m], pa[0][2 * m + 1], pa[1][2 * m + 1], b0, b1);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j] += e[j];
            if constexpr (FMT == kFmtInt4) {
                const bool hi = ((ub0 + bk) & 1) != 0;
                const uint32_t w0 = rs[(slot * 2 + 0) * 32 + lane], w1 = rs[(slot * 2 + 1) * 32 + lane];
                const float sc0 = __uint_as_float(hi ? (w0 & 0xFFFF0000u) : (w0 << 16));
                const float sc1 = __uint_as_float(hi ? (w1 & 0xFFFF0000u) : (w1 << 16));
                cur[0] = fmaf(d[0], sc0, cur[0]);
                cur[1] = fmaf(d[1], sc0, cur[1]);
                cur[2] = fmaf(d[2], sc1, cur[2]);
                cur[3] = fmaf(d[3], sc1, cur[3]);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) cur[j] += d[j];
            }
            if (++slot == kRD) slot = 0;
            if (++bk == nblk) {  // the tile's part is done: into its accumulators
#pragma unroll
                for (int ii = 0; ii < kTPW; ++ii)
                    if (ii == i) {
#pragma unroll
                        for (int j = 0; j < 4; ++j) acc[ii][j] += cur[j];
                    }
#pragma unroll
                for (int j = 0; j < 4; ++j) cur[j] = 0.f;
                bk = 0;
                ++i;
            }
        }
        cp_async_wait<0>();
    }

    // ---- the K parts of a tile meet in shared memory (the staging area is free now)
    if (ks > 1) {
        __syncthreads();
        float *red2 = reinterpret_cast<float *>(sx);  // [kNW][kTPW][4][32]
#pragma unroll
        for (int i = 0; i < kTPW; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) red2[((warp * kTPW + i) * 4 + j) * 32 + lane] = acc[i][j];
        __syncthreads();
        if (kp == 0) {
#pragma unroll
            for (int i = 0; i < kTPW; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    for (int q = 1; q < ks; ++q) acc[i][j] += red2[(((warp + q) * kTPW + i) * 4 + j) * 32 + lane];
        }
    }
    if (kp != 0) return;

    // ---- epilogue: lane (g, t) holds rows (g, g + 8) x sequences (2t, 2t + 1)
#pragma unroll
    for (int i = 0; i < kTPW; ++i) {
        const int ti = gw + i * nwarps;
        if (ti >= tiles) break;
        const uint4 *r0, *r1;
        const void *s0, *s1;
        int rr0, rr1;
        row_ptrs(ti, r0, r1, s0, s1, rr0, rr1);
        float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
        if constexpr (FMT == kFmtInt8) {
            const float sa = __ldg(static_cast<const float *>(s0) + rr0), sb = __ldg(static_cast<const float *>(s1) + rr1);
            v[0] *= sa;
            v[1] *= sa;
            v[2] *= sb;
            v[3] *= sb;
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int b = 2 * t + c;
            if (b >= B) continue;
            if (a.mode == 2) {
                const float gt = v[c], up = v[2 + c];
                a.y[(size_t)b * a.ldy + ti * 8 + g] = gt / (1.f + __expf(-gt)) * up;
                continue;
            }
            const int row0 = ti * 16 + g, row1 = row0 + 8;
            float y0 = v[c], y1 = v[2 + c];
            if (a.mode == 0) {
                int seg = 0, r = row0;
                while (seg + 1 < a.n_seg && r >= a.seg_rows[seg]) r -= a.seg_rows[seg++];
                if (a.bias[seg]) {
                    y0 += bf16_bits_to_float(__ldg(a.bias[seg] + r));
                    y1 += bf16_bits_to_float(__ldg(a.bias[seg] + r + 8));
                }
            }
            float *yb = a.y + (size_t)b * a.ldy;
            if (a.mode == 1 && gridDim.y > 1) {  // the K parts of other CTAs add into the same rows
                atomicAdd(yb + row0, y0);
                atomicAdd(yb + row1, y1);
            } else if (a.mode == 1) {
                yb[row0] += y0;
                yb[row1] += y1;
            } else {
                yb[row0] = y0;
                yb[row1] = y1;
            }
        }
    }
}

// ---- small per-sequence kernels ---------------------------------------------

// x[b] = embedding row of token st[b].token.
__global__ void k_bembed(const uint16_t *embed, const DevState *st, int B, int h, float *x) {
    const int b = blockIdx.x;
    const int tok = st[b].token;
    for (int i = threadIdx.x; i < h; i += blockDim.x)
        x[(size_t)b * h + i] = bf16_bits_to_float(embed[(size_t)tok * h + i]);
}

// Per (sequence, head) of the raw QKV rows: optional RMSNorm of q and k heads,
// RoPE at the sequence's position, q into q_out, K and V rounded to bf16 and
// written at slot pos % 16 of the sequence's page table[pos / 16].
__global__ void k_bqkv_post(BQkvPostArgs a) {
    const int b = blockIdx.y, head = blockIdx.x, lane = threadIdx.x;
    if (a.part && !a.part[b]) return;
    const int H = a.Hq + 2 * a.Hkv, d = a.d, half = d / 2;
    const int pos = a.st[b].pos;
    const float *raw = a.raw + (size_t)b * H * d + (size_t)head * d;
    const bool is_q = head < a.Hq, is_k = !is_q && head < a.Hq + a.Hkv;
    float v[4];  // lane holds elements lane + 32 m (d <= 128)
    const int M = d / 32;
#pragma unroll
    for (int m = 0; m < 4; ++m) v[m] = m < M ? raw[lane + 32 * m] : 0.f;
    if ((is_q || is_k) && a.q_gain) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) ss += v[m] * v[m];
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / (float)d + a.eps);
        const uint16_t *gm = is_q ? a.q_gain : a.k_gain;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (m < M) v[m] = bf16_bits_to_float(gm[lane + 32 * m]) * (v[m] * inv);
    }
    if (is_q || is_k) {  // rotate pairs (i, i + d/2) by pos * theta_i
        const float2 *cs = a.rope_cs + (size_t)pos * half;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            if (m >= M / 2) break;
            const float2 c = cs[lane + 32 * m];
            const float x0 = v[m], x1 = v[m + M / 2];
            v[m] = x0 * c.x - x1 * c.y;
            v[m + M / 2] = x1 * c.x + x0 * c.y;
        }
    }
    if (is_q) {
        float *q = a.q_out + (size_t)b * a.Hq * d + (size_t)head * d;
#pragma unroll
        for (int m = 0; m < 4; ++m)
            if (m < M) q[lane + 32 * m] = v[m];
        return;
    }
    const int gk = is_k ? head - a.Hq : head - a.Hq - a.Hkv;
    int phys = a.page_table[(size_t)b * a.max_pages + pos / kPageTokens];
    if (phys < 0 || phys >= a.n_pages) {
        if (lane == 0) atomicCAS(&a.st[b].err, kErrNone, kErrBadPage);
        return;
    }
    uint16_t *dst = (is_k ? a.k_pool : a.v_pool) + ((((size_t)phys * a.Hkv + gk) * kPageTokens) + pos % kPageTokens) * d;
#pragma unroll
    for (int m = 0; m < 4; ++m)
        if (m < M) dst[lane + 32 * m] = float_to_bf16_bits(v[m]);
}

// Greedy argmax per sequence (lowest index on ties) in two steps: CTA (x, b)
// reduces its slice of sequence b's logits to one (value, index) pair; then one
// warp per sequence reduces the pairs and, for the sequences taking part in the
// step, makes the token the next input and moves the position on.
constexpr int kArgSplits = 32;
__global__ void k_bargmax_part(const float *logits, int V, float *pv, int *pi) {
    const int b = blockIdx.y, sp = blockIdx.x;
    const int lo = (int)((long long)V * sp / kArgSplits), hi = (int)((long long)V * (sp + 1) / kArgSplits);
    const float *lg = logits + (size_t)b * V;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int i = lo + threadIdx.x; i < hi; i += blockDim.x) {
        const float v = lg[i];
        if (v > best || (v == best && i < bi)) {
            best = v;
            bi = i;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) {
            best = ov;
            bi = oi;
        }
    }
    __shared__ float sv[32];
    __shared__ int si[32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        sv[warp] = best;
        si[warp] = bi;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
            if (sv[w] > best || (sv[w] == best && si[w] < bi)) {
                best = sv[w];
                bi = si[w];
            }
        pv[b * kArgSplits + sp] = best;
        pi[b * kArgSplits + sp] = bi;
    }
}

__global__ void k_bargmax_final(const float *pv, const int *pi, DevState *st, const int *part) {
    const int b = blockIdx.x, lane = threadIdx.x;
    float best = pv[b * kArgSplits + lane];
    int bi = pi[b * kArgSplits + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) {
            best = ov;
            bi = oi;
        }
    }
    if (lane == 0) {
        st[b].last_token = bi;
        if (!part || part[b]) {
            st[b].token = bi;
            st[b].pos += 1;
        }
    }
}

template <int FMT>
cudaError_t launch_fmt(const LaunchCfg &lc, const BGemvArgs &a, int grid, int gks) {
    // staging for min(K part, kKC) values of 8 sequences (it also holds the K-part sums), then
    // the warps' weight rings
    int stage_entries = (a.K + gks - 1) / gks + 128;
    if (stage_entries > kKC) stage_entries = kKC;
    if (stage_entries < kRedEntries) stage_entries = kRedEntries;
    const size_t smem = (size_t)stage_entries * 16 + (size_t)kNW * kRingWarpBytes;
    if (smem > (size_t)kMaxSmemOptin) return cudaErrorInvalidValue;
    return launch_k(lc, k_bgemv<FMT>, dim3(grid, gks), dim3(kNW * 32), smem, a);
}

}  // namespace

bool bgemv_shape_ok(int fmt, int N, int K, int mode) {
    // INT4: K % 256 (an even number of groups per row: a block's parity picks its scale's half)
    const int blk = fmt == kFmtInt4 ? 256 : (fmt == kFmtInt8 ? 64 : 32);
    return K > 0 && K % blk == 0 && K % 8 == 0 && N > 0 && N % (mode == 2 ? 8 : 16) == 0;
}

// K split: as many warps per tile (a divisor of kNW) as it takes for the tiles to give every
// warp of the grid work; then the grid, at most kTPW tiles per tile slot.
// Large-K projections that add into y (the down projection) also split K over
// grid.y CTAs of about 2048 values each, so that a CTA stages only its part of the
// inputs; their partial sums meet in y through atomic adds.
void bgemv_plan(const LaunchCfg &lc, int N, int K, int mode, int &ks, int &grid, int &gks) {
    const int tiles = mode == 2 ? N / 8 : N / 16;
    gks = 1;
    if (mode == 1 && K > kNormK) {
        gks = K / 2048;
        if (gks > 8) gks = 8;
    }
    const int n_sm = lc.n_sm / gks > 0 ? lc.n_sm / gks : 1;  // SMs per K part
    // the smallest divisor of kNW that gives every warp of the grid work, else the largest
    ks = 1;
    for (int d = 1; d <= kNW; ++d) {
        if (kNW % d) continue;
        ks = d;
        if ((long long)tiles * d >= (long long)kNW * n_sm) break;
    }
    const int tslots = kNW / ks;
    grid = (tiles + tslots - 1) / tslots;
    if (grid > n_sm) grid = n_sm;
    while ((long long)grid * tslots * kTPW < tiles) ++grid;
}

cudaError_t launch_bgemv(const LaunchCfg &lc, int fmt, const BGemvArgs &args) {
    if (args.B < 1 || args.B > 8 || !bgemv_shape_ok(fmt, args.N, args.K, args.mode) ||
        (args.gamma && args.K > kNormK))
        return cudaErrorInvalidValue;
    BGemvArgs a = args;
    int grid = 0, gks = 1;
    bgemv_plan(lc, a.N, a.K, a.mode, a.ks, grid, gks);
    if (fmt == kFmtInt4) return launch_fmt<kFmtInt4>(lc, a, grid, gks);
    if (fmt == kFmtInt8) return launch_fmt<kFmtInt8>(lc, a, grid, gks);
    if (fmt == kFmtBf16) return launch_fmt<kFmtBf16>(lc, a, grid, gks);
    return cudaErrorInvalidValue;
}

cudaError_t launch_bembed(cudaStream_t s, const uint16_t *embed, const DevState *st, int B, int h, float *x) {
    k_bembed<<<B, 256, 0, s>>>(embed, st, B, h, x);
    return cudaGetLastError();
}

cudaError_t launch_bqkv_post(cudaStream_t s, const BQkvPostArgs &a, int B) {
    if (a.d != 64 && a.d != 128) return cudaErrorInvalidValue;
    k_bqkv_post<<<dim3(a.Hq + 2 * a.Hkv, B), 32, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_bargmax(cudaStream_t s, const float *logits, int V, DevState *st, int B, const int *part,
                           float *pv, int *pi) {
    static_assert(kArgSplits == 32, "one lane per split in the final step");
    k_bargmax_part<<<dim3(kArgSplits, B), 256, 0, s>>>(logits, V, pv, pi);
    k_bargmax_final<<<B, 32, 0, s>>>(pv, pi, st, part);
    return cudaGetLastError();
}

}  // namespace qd
