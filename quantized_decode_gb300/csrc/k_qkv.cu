// k_qkv.cu - fused RMSNorm -> Q/K/V dequant GEMV (+bias) -> (per-head q/k RMSNorm)
// -> RoPE -> paged KV append, one kernel per layer of the decode step.
//
// Rows of the three projections are numbered q | k | v; warps stream tiles of
// TR rows (gemv_stream).  A tile never straddles a head (TR divides d).
// Without per-head q/k norms, a lane's two rows are the RoPE pair (p, p + d/2)
// of one head (a tile holds pairs p0 .. p0 + 3), so the tile's epilogue
// rotates them at the current position and writes q to the query buffer or
// k/v rounded to bf16 into slot pos % 16 of page page_table[pos / 16] at once.
// With the norms (Qwen3) a head's RMS needs all its rows: tiles hold 8
// consecutive rows, and the warp that completes the last tile of a head
// (per-head arrival counter) runs that head's epilogue: RMSNorm, RoPE, write.
#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kRT = 2;  // rows per lane (a RoPE pair in the pair tiling)
// ring depth: INT4 rows 2 (copies 1 step ahead; measured: 8.8 us against 9.3 at D = 5),
// INT8 rows 5 (a step covers half the K values)
template <int FMT>
constexpr int kQD = FMT == kFmtInt4 ? 2 : 5;

template <int D>
QD_DEV void head_epilogue(const QkvArgs &a, int head, int pos, int lane) {
    constexpr int M = D / 32;
    float v[M];
    const float *raw = a.raw + (size_t)head * D;
#pragma unroll
    for (int m = 0; m < M; ++m) v[m] = __ldcg(raw + lane + 32 * m);
    const bool is_q = head < a.Hq;
    const bool is_k = !is_q && head < a.Hq + a.Hkv;
    if ((is_q || is_k) && a.q_gain) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) ss += v[m] * v[m];
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / (float)D + a.eps);
        const uint16_t *g = is_q ? a.q_gain : a.k_gain;
#pragma unroll
        for (int m = 0; m < M; ++m) v[m] = bf16_bits_to_float(__ldg(g + lane + 32 * m)) * (v[m] * inv);
    }
    if (is_q || is_k) {
        const float2 *cs = a.rope_cs + (size_t)pos * (D / 2);
#pragma unroll
        for (int m = 0; m < M / 2; ++m) {
            const float2 c = __ldg(cs + lane + 32 * m);
            const float x0 = v[m], x1 = v[m + M / 2];
            v[m] = x0 * c.x - x1 * c.y;
            v[m + M / 2] = x1 * c.x + x0 * c.y;
        }
    }
    if (is_q) {
#pragma unroll
        for (int m = 0; m < M; ++m) a.q_out[(size_t)head * D + lane + 32 * m] = v[m];
        return;
    }
    const int g = is_k ? head - a.Hq : head - a.Hq - a.Hkv;
    const int phys = a.page_table[pos / kPageTokens];
    if (phys < 0 || phys >= a.n_pages) {
        if (lane == 0) atomicCAS(&a.st->err, kErrNone, kErrBadPage);
        return;
    }
    uint16_t *dst = (is_k ? a.k_pool : a.v_pool) +
                    (((size_t)phys * a.Hkv + g) * kPageTokens + pos % kPageTokens) * D;
    uint16_t *cpy = a.kv_new ? a.kv_new + ((size_t)(is_k ? 0 : a.Hkv) + g) * D : nullptr;
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const uint16_t b = float_to_bf16_bits(v[m]);
        dst[lane + 32 * m] = b;
        if (cpy) cpy[lane + 32 * m] = b;
    }
}

// The static inputs of a RoPE pair's epilogue: bias, INT8 row scales and the
// (cos, sin) of pair p at position pos.  Loaded before the dependency wait for
// a warp's first tiles, so that the epilogue does not wait on them.
struct PairConst {
    float b0, b1, s0, s1;
    float2 cs;
};
template <int FMT, int D>
QD_DEV PairConst pair_const(const QkvArgs &a, int head, int p, int r0, int pos) {
    const int seg = head < a.Hq ? 0 : (head < a.Hq + a.Hkv ? 1 : 2);
    const int base = seg == 0 ? 0 : (seg == 1 ? a.rows_q : a.rows_q + a.rows_kv);
    const int l0 = r0 - base, l1 = l0 + D / 2;
    PairConst c{0.f, 0.f, 1.f, 1.f, make_float2(1.f, 0.f)};
    if constexpr (FMT == kFmtInt8) {
        c.s0 = __ldg((const float *)a.s[seg] + l0);
        c.s1 = __ldg((const float *)a.s[seg] + l1);
    }
    if (a.b[seg]) {
        c.b0 = bf16_bits_to_float(__ldg(a.b[seg] + l0));
        c.b1 = bf16_bits_to_float(__ldg(a.b[seg] + l1));
    }
    if (seg < 2) c.cs = __ldg(a.rope_cs + (size_t)pos * (D / 2) + p);
    return c;
}

// Rows (p, p + D/2) of head `head` (global row r0 = head * D + p): scale, bias,
// RoPE for q and k at position pos, then q out or the bf16 K/V append.
template <int FMT, int D>
QD_DEV void pair_epilogue(const QkvArgs &a, int head, int p, const float (&out)[2], float post, int pos,
                          int phys, const PairConst &c) {
    const int seg = head < a.Hq ? 0 : (head < a.Hq + a.Hkv ? 1 : 2);
    float v0 = out[0] * post * c.s0 + c.b0, v1 = out[1] * post * c.s1 + c.b1;
    if (seg < 2) {
        const float x0 = v0, x1 = v1;
        v0 = x0 * c.cs.x - x1 * c.cs.y;
        v1 = x1 * c.cs.x + x0 * c.cs.y;
    }
    if (seg == 0) {
        a.q_out[(size_t)head * D + p] = v0;
        a.q_out[(size_t)head * D + p + D / 2] = v1;
        return;
    }
    const int g = head - a.Hq - (seg == 2 ? a.Hkv : 0);
    if (phys < 0 || phys >= a.n_pages) {
        atomicCAS(&a.st->err, kErrNone, kErrBadPage);
        return;
    }
    uint16_t *dst = (seg == 1 ? a.k_pool : a.v_pool) + (((size_t)phys * a.Hkv + g) * kPageTokens + pos % kPageTokens) * D;
    const uint16_t b0 = float_to_bf16_bits(v0), b1 = float_to_bf16_bits(v1);
    dst[p] = b0;
    dst[p + D / 2] = b1;
    if (a.kv_new) {
        uint16_t *cpy = a.kv_new + ((size_t)(seg == 1 ? 0 : a.Hkv) + g) * D;
        cpy[p] = b0;
        cpy[p + D / 2] = b1;
    }
}

constexpr int kMaxWarps = 12;
constexpr int kLPR = kLanesPerRow;

template <int FMT, int DH>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) k_qkv(QkvArgs a) {
    TimelineMark timeline_mark{a.tl};
    l2_prefetch_share(a.pf, blockIdx.x, gridDim.x);
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    constexpr int S = 32 / kLPR;
    constexpr int TR = S * kRT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / kLPR, j = lane % kLPR;
    const int NW = blockDim.x >> 5, ks = a.ks, tpc = NW / ks;
    const int kp = warp % ks, tslot = warp / ks;
    const int NP = slabs_per_row(FMT, a.K);
    const int U = units_per_row(FMT, a.K);
    const int PP = (NP + ks - 1) / ks;
    const int p_begin = kp * PP, p_end = min(NP, p_begin + PP);
    const int rows_total = a.rows_q + 2 * a.rows_kv;
    const size_t rb = FMT == kFmtInt4 ? (size_t)a.K / 2 : (size_t)a.K;
    const int G = a.K / kGroup;
    half2 *xs = reinterpret_cast<half2 *>(smem);
    const size_t xbytes = ((size_t)a.K * 2 + 15) & ~(size_t)15;
    uint16_t *gs = reinterpret_cast<uint16_t *>((char *)smem + xbytes);  // the attention norm's gain
    uint4 *ring;
    uint32_t *sring;
    warp_rings<kRT, kQD<FMT>>((char *)smem + 2 * xbytes, NW, warp, ring, sring);
    float *kred = reinterpret_cast<float *>((char *)smem + 2 * xbytes + (size_t)NW * ring_bytes_per_warp<kRT, kQD<FMT>>()) +
                  (size_t)tslot * ks * 32 * kRT;
    float post = 1.f;
    int pos = 0, phys = -1;
    PairConst pc[2];  // the lane's first two tiles (pair mode; j == 0 lanes of the reducing warp)
    // pair mode: tile t = pairs (t % TPH) * S .. + S - 1 of head t / TPH
    const bool pairs = a.q_gain == nullptr;
    constexpr int TPH = DH / TR;

    auto segment = [&](int r, int &seg, int &local) {
        seg = r < a.rows_q ? 0 : (r < a.rows_q + a.rows_kv ? 1 : 2);
        local = r - (seg == 0 ? 0 : (seg == 1 ? a.rows_q : a.rows_q + a.rows_kv));
    };
    // global row of row i of this lane's slot in tile t
    auto row_of = [&](int t, int i) -> int {
        if (pairs) return (t / TPH) * DH + (t % TPH) * S + slot + i * (DH / 2);
        return t * TR + slot * kRT + i;
    };
    auto rows = [&](int t, int i) -> RowRef {
        int seg, local;
        segment(row_of(t, i), seg, local);
        return {reinterpret_cast<const uint4 *>((const char *)a.w[seg] + (size_t)local * rb),
                (const uint16_t *)a.s[seg] + (size_t)local * G};
    };
    const int t_first = blockIdx.x * tpc + tslot, t_stride = gridDim.x * tpc, n_tiles = rows_total / TR;
    auto sync = [&]() {
        cp_async_wait<kQD<FMT> - 1>();  // the gain (the ring's first steps stay in flight)
        // static data and the position (final: the step's first kernel starts after the last step)
        pos = __ldcg(&a.st->pos);
        if (pairs && j == 0 && kp == 0) {
            const int t0 = t_first, t1 = t_first + t_stride;
            if (t0 < n_tiles) pc[0] = pair_const<FMT, DH>(a, t0 / TPH, (t0 % TPH) * S + slot, row_of(t0, 0), pos);
            if (t1 < n_tiles) pc[1] = pair_const<FMT, DH>(a, t1 / TPH, (t1 % TPH) * S + slot, row_of(t1, 0), pos);
        }
        pdl_wait();
        const uint16_t *erow = a.embed ? a.embed + (size_t)__ldcg(&a.st->token) * a.K : nullptr;
        if (erow && blockIdx.x == 0)
            for (int i = threadIdx.x; i < a.K; i += blockDim.x) a.x_init[i] = bf16_bits_to_float(erow[i]);
        post = stage_activations(a.x, erow, a.gamma, a.eps, a.K, erow ? nullptr : a.stats_in, xs, nullptr, red,
                                 act_blk_bytes<FMT>(), gs, nullptr, nullptr, nullptr, erow ? nullptr : a.x2);
        phys = __ldg(a.page_table + pos / kPageTokens);  // used by the k/v tiles' epilogues
        pdl_launch();
    };
    auto epi = [&](int t, float(&out)[kRT]) {
        if (!ksplit_reduce<kRT>(out, ks, kp, tslot, kred, j, slot, kLPR)) return;
        if (pairs) {
            if (j != 0) return;
            const int k = (t - t_first) / t_stride;
            const PairConst c = k == 0   ? pc[0]
                                : k == 1 ? pc[1]
                                         : pair_const<FMT, DH>(a, t / TPH, (t % TPH) * S + slot, row_of(t, 0), pos);
            pair_epilogue<FMT, DH>(a, t / TPH, (t % TPH) * S + slot, out, post, pos, phys, c);
            return;
        }
        const int tile_r = t * TR;
        int seg, local;
        segment(tile_r, seg, local);
        local += slot * kRT;
        if (j == 0) {
#pragma unroll
            for (int i = 0; i < kRT; ++i) {
                float v = out[i] * post;
                if constexpr (FMT == kFmtInt8) v *= __ldg((const float *)a.s[seg] + local + i);
                if (a.b[seg]) v += bf16_bits_to_float(__ldg(a.b[seg] + local + i));
                a.raw[tile_r + slot * kRT + i] = v;
            }
        }
        __threadfence();
        __syncwarp();
        const int head = tile_r / DH;
        int last = 0;
        if (lane == 0) last = (atomicAdd(&a.head_cnt[head], TR) + TR == DH);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            head_epilogue<DH>(a, head, pos, lane);
            if (lane == 0) a.head_cnt[head] = 0;
        }
    };
    gain_copy_async(a.gamma, a.K, gs);
    gemv_stream<FMT, kRT, kQD<FMT>>(rows, epi, sync, t_first, t_stride, n_tiles, p_begin, p_end, U, j, xs, ring, sring);
}

template <int FMT, int DH>
cudaError_t launch_qkv_d(const LaunchCfg &lc, QkvArgs a) {
    const int rows = a.rows_q + 2 * a.rows_kv;
    const int tiles = rows / ((32 / kLPR) * kRT);
    const int NP = slabs_per_row(FMT, a.K);
    int ks = 1;
    while (ks < 4 && tiles * ks < 8 * lc.n_sm && NP / (ks * 2) >= 1) ks *= 2;
    GemvPlan pl = plan_gemv(tiles, ks, lc.n_sm, kMaxWarps);
    a.ks = ks;
    const size_t smem = 2 * (((size_t)a.K * 2 + 15) & ~(size_t)15) + (size_t)pl.nw * ring_bytes_per_warp<kRT, kQD<FMT>>() +
                        (size_t)pl.nw * 32 * kRT * 4;
    return launch_k(lc, k_qkv<FMT, DH>, dim3(pl.grid), dim3(pl.nw * 32), smem, a);
}

}  // namespace

bool qkv_shape_ok(int fmt, int rows_q, int rows_kv, int K, int d) {
    if (d != 64 && d != 128) return false;
    if (fmt == kFmtInt4 ? (K % 256 != 0) : (K % 128 != 0)) return false;
    const int U = fmt == kFmtInt4 ? K / 32 : K / 16;
    const int lpr = pick_lpr(U);
    if (!lpr) return false;
    const int TR = (32 / lpr) * kRT;
    return d % TR == 0 && rows_q % d == 0 && rows_kv % d == 0 && (size_t)K * 2 <= 200 * 1024;
}

cudaError_t launch_qkv(const LaunchCfg &lc, int fmt, const QkvArgs &a) {
    if (fmt == kFmtInt4) return a.d == 128 ? launch_qkv_d<kFmtInt4, 128>(lc, a) : launch_qkv_d<kFmtInt4, 64>(lc, a);
    if (fmt == kFmtInt8) return a.d == 128 ? launch_qkv_d<kFmtInt8, 128>(lc, a) : launch_qkv_d<kFmtInt8, 64>(lc, a);
    return cudaErrorInvalidValue;
}

}  // namespace qd
