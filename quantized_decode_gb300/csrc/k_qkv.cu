// k_qkv.cu - fused RMSNorm -> Q/K/V dequant GEMV (+bias) -> (per-head q/k RMSNorm)
// -> RoPE -> paged KV append, one kernel per layer of the decode step.
//
// Rows of the three projections are numbered q | k | v; warps take tiles of
// TR rows round-robin.  A tile never straddles a head (TR divides d), so the
// warp that completes the last tile of a head (per-head arrival counter) runs
// that head's epilogue: per-head RMSNorm (Qwen3), RoPE with pairs (i, i+d/2)
// at the current position, then q to the query buffer or k/v rounded to bf16
// into slot pos % 16 of page page_table[pos / 16].
#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kNT = 256;
constexpr int kRT = 4;

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
#pragma unroll
    for (int m = 0; m < M; ++m) dst[lane + 32 * m] = float_to_bf16_bits(v[m]);
}

template <int FMT, int LPR, int D>
__global__ void __launch_bounds__(kNT) k_qkv(QkvArgs a) {
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    constexpr int S = 32 / LPR;
    constexpr int TR = S * kRT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LPR, j = lane % LPR;
    const int rows_total = a.rows_q + 2 * a.rows_kv;
    const int n_tiles = rows_total / TR;
    const int W = gridDim.x * (kNT / 32);
    const int U = FMT == kFmtInt4 ? a.K / 32 : a.K / 16;
    const size_t row_bytes = FMT == kFmtInt4 ? (size_t)a.K / 2 : (size_t)a.K;

    // Weights do not depend on earlier kernels: warm L2 with this warp's first tile.
    {
        const int t = blockIdx.x * (kNT / 32) + warp;
        if (t < n_tiles) {
            const int r = t * TR;
            const int seg = r < a.rows_q ? 0 : (r < a.rows_q + a.rows_kv ? 1 : 2);
            const int local = r - (seg == 0 ? 0 : (seg == 1 ? a.rows_q : a.rows_q + a.rows_kv));
            const char *base = (const char *)a.w[seg] + (size_t)local * row_bytes;
            for (size_t off = (size_t)lane * 128; off < TR * row_bytes; off += 32 * 128)
                prefetch_l2(base + off);
        }
    }

    pdl_wait();
    const int pos = a.st->pos;
    const int token = a.st->token;
    const uint16_t *erow = a.embed ? a.embed + (size_t)token * a.K : nullptr;
    if (erow && blockIdx.x == 0) {
        for (int i = threadIdx.x; i < a.K; i += kNT) a.x_init[i] = bf16_bits_to_float(erow[i]);
    }
    half2 *xs = reinterpret_cast<half2 *>(smem);
    const float post = stage_activations<kNT>(a.x, erow, a.gamma, a.eps, a.K, xs, nullptr, red);
    pdl_launch();

    for (int t = blockIdx.x * (kNT / 32) + warp; t < n_tiles; t += W) {
        const int tile_r = t * TR;
        const int r0 = tile_r + slot * kRT;
        const int seg = tile_r < a.rows_q ? 0 : (tile_r < a.rows_q + a.rows_kv ? 1 : 2);
        const int seg0 = seg == 0 ? 0 : (seg == 1 ? a.rows_q : a.rows_q + a.rows_kv);
        const int local = r0 - seg0;
        const uint4 *wrow[kRT];
        float out[kRT];
        if constexpr (FMT == kFmtInt4) {
            const uint16_t *srow[kRT];
#pragma unroll
            for (int i = 0; i < kRT; ++i) {
                wrow[i] = reinterpret_cast<const uint4 *>((const char *)a.w[seg] + (size_t)(local + i) * row_bytes);
                srow[i] = (const uint16_t *)a.s[seg] + (size_t)(local + i) * (a.K / kGroup);
            }
            int4_tile_dots<LPR, kRT>(wrow, srow, reinterpret_cast<const uint4 *>(xs), U, j, out);
        } else {
#pragma unroll
            for (int i = 0; i < kRT; ++i)
                wrow[i] = reinterpret_cast<const uint4 *>((const char *)a.w[seg] + (size_t)(local + i) * row_bytes);
            int8_tile_dots<LPR, kRT>(wrow, reinterpret_cast<const uint4 *>(xs), U, j, out);
#pragma unroll
            for (int i = 0; i < kRT; ++i) out[i] *= __ldg((const float *)a.s[seg] + local + i);
        }
        if (j == 0) {
#pragma unroll
            for (int i = 0; i < kRT; ++i) {
                float v = out[i] * post;
                if (a.b[seg]) v += bf16_bits_to_float(__ldg(a.b[seg] + local + i));
                a.raw[r0 + i] = v;
            }
        }
        __threadfence();
        __syncwarp();
        const int head = tile_r / D;
        int last = 0;
        if (lane == 0) last = (atomicAdd(&a.head_cnt[head], TR) + TR == D);
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            head_epilogue<D>(a, head, pos, lane);
            if (lane == 0) a.head_cnt[head] = 0;
        }
    }
}

template <int FMT, int D>
cudaError_t launch_qkv_d(const LaunchCfg &lc, const QkvArgs &a) {
    const int U = FMT == kFmtInt4 ? a.K / 32 : a.K / 16;
    const int lpr = pick_lpr(U);
    const size_t smem = (size_t)a.K * sizeof(__half);
    const int rows = a.rows_q + 2 * a.rows_kv;
    const int tiles = rows / ((32 / lpr) * kRT);
    int grid = (tiles + kNT / 32 - 1) / (kNT / 32);
    if (grid > 2 * lc.n_sm) grid = 2 * lc.n_sm;
    switch (lpr) {
        case 32: return launch_k(lc, k_qkv<FMT, 32, D>, dim3(grid), dim3(kNT), smem, a);
        case 16: return launch_k(lc, k_qkv<FMT, 16, D>, dim3(grid), dim3(kNT), smem, a);
        case 8: return launch_k(lc, k_qkv<FMT, 8, D>, dim3(grid), dim3(kNT), smem, a);
        default: return cudaErrorInvalidValue;
    }
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
