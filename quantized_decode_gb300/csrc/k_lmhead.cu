// k_lmhead.cu - final RMSNorm -> LM-head GEMV -> logits + fused greedy argmax.
//
// Each CTA stages RMSNorm(x) once, streams its rows (bf16, or INT8 with a row
// scale) and keeps the running (max, lowest index) pair; the CTA's pair goes to
// a per-CTA slot, and the CTA that arrives last (arrival counter, no waiting)
// reduces the slots, writes the token and, inside the decode step, hands it to
// the next step as input and advances the position.
#include <climits>

#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kNT = 256;
constexpr int kRT = 4;

QD_DEV void better(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

template <int FMT, int LPR>
__global__ void __launch_bounds__(kNT) k_lm_head(LmHeadArgs a) {
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    __shared__ float s_val[kNT / 32];
    __shared__ int s_idx[kNT / 32];
    __shared__ int s_last;
    constexpr int S = 32 / LPR;
    constexpr int TR = S * kRT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LPR, j = lane % LPR;
    const int U = FMT == kFmtBf16 ? a.K / 8 : a.K / 16;
    const size_t row_bytes = FMT == kFmtBf16 ? (size_t)a.K * 2 : (size_t)a.K;
    const int n_tiles = a.N / TR;
    const int W = gridDim.x * (kNT / 32);

    {
        const int t = blockIdx.x * (kNT / 32) + warp;
        if (t < n_tiles) {
            const char *base = (const char *)a.w + (size_t)t * TR * row_bytes;
            for (size_t off = (size_t)lane * 128; off < TR * row_bytes; off += 32 * 128) prefetch_l2(base + off);
        }
    }

    pdl_wait();
    float post;
    if constexpr (FMT == kFmtBf16)
        post = stage_activations<kNT>(a.x, nullptr, a.gamma, a.eps, a.K, nullptr,
                                      reinterpret_cast<float *>(smem), red);
    else
        post = stage_activations<kNT>(a.x, nullptr, a.gamma, a.eps, a.K,
                                      reinterpret_cast<half2 *>(smem), nullptr, red);
    pdl_launch();

    float best = -INFINITY;
    int bidx = INT_MAX;
    for (int t = blockIdx.x * (kNT / 32) + warp; t < n_tiles; t += W) {
        const int r0 = t * TR + slot * kRT;
        const uint4 *wrow[kRT];
#pragma unroll
        for (int i = 0; i < kRT; ++i)
            wrow[i] = reinterpret_cast<const uint4 *>((const char *)a.w + (size_t)(r0 + i) * row_bytes);
        float out[kRT];
        if constexpr (FMT == kFmtBf16) {
            bf16_tile_dots<LPR, kRT>(wrow, reinterpret_cast<const float4 *>(smem), U, j, out);
        } else {
            int8_tile_dots<LPR, kRT>(wrow, smem, U, j, out);
#pragma unroll
            for (int i = 0; i < kRT; ++i) out[i] *= __ldg(a.scale + r0 + i);
        }
        if (j == 0) {
#pragma unroll
            for (int i = 0; i < kRT; ++i) {
                const float v = out[i] * post;
                a.logits[r0 + i] = v;
                better(best, bidx, v, r0 + i);
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bidx, o);
        better(best, bidx, v2, i2);
    }
    if (lane == 0) {
        s_val[warp] = best;
        s_idx[warp] = bidx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kNT / 32; ++w) better(best, bidx, s_val[w], s_idx[w]);
        a.part_val[blockIdx.x] = best;
        a.part_idx[blockIdx.x] = bidx;
        __threadfence();
        s_last = atomicAdd(a.counter, 1) == (int)gridDim.x - 1;
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    best = -INFINITY;
    bidx = INT_MAX;
    for (int c = threadIdx.x; c < (int)gridDim.x; c += kNT) better(best, bidx, __ldcg(a.part_val + c), __ldcg(a.part_idx + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bidx, o);
        better(best, bidx, v2, i2);
    }
    if (lane == 0) {
        s_val[warp] = best;
        s_idx[warp] = bidx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < kNT / 32; ++w) better(best, bidx, s_val[w], s_idx[w]);
        int tok = bidx;
        if (tok < 0 || tok >= a.N) {  // every logit was NaN
            tok = 0;
            if (a.st) atomicCAS(&a.st->err, kErrNone, kErrBadToken);
        }
        *a.token_out = tok;
        if (a.st) {
            a.st->last_token = tok;
            a.st->token = tok;
            if (a.advance) a.st->pos += 1;
        }
        *a.counter = 0;
    }
}

template <int FMT>
cudaError_t launch_fmt(const LaunchCfg &lc, const LmHeadArgs &a, int grid) {
    const int U = FMT == kFmtBf16 ? a.K / 8 : a.K / 16;
    const int lpr = pick_lpr(U);
    const size_t smem = FMT == kFmtBf16 ? (size_t)a.K * 4 : (size_t)a.K * 2;
    switch (lpr) {
        case 32: return launch_k(lc, k_lm_head<FMT, 32>, dim3(grid), dim3(kNT), smem, a);
        case 16: return launch_k(lc, k_lm_head<FMT, 16>, dim3(grid), dim3(kNT), smem, a);
        case 8: return launch_k(lc, k_lm_head<FMT, 8>, dim3(grid), dim3(kNT), smem, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool lm_head_shape_ok(int fmt, int N, int K) {
    if (fmt != kFmtBf16 && fmt != kFmtInt8) return false;
    if (K % 256 != 0 || (size_t)K * 4 > 200 * 1024) return false;
    const int U = fmt == kFmtBf16 ? K / 8 : K / 16;
    const int lpr = pick_lpr(U);
    return lpr && N > 0 && N % ((32 / lpr) * kRT) == 0;
}

int lm_head_grid(const LaunchCfg &lc, int N) {
    const int tiles = N / kRT;
    int grid = (tiles + kNT / 32 - 1) / (kNT / 32);
    if (grid > 2 * lc.n_sm) grid = 2 * lc.n_sm;
    return grid < 1 ? 1 : grid;
}

cudaError_t launch_lm_head(const LaunchCfg &lc, const LmHeadArgs &a, int grid) {
    if (a.fmt == kFmtBf16) return launch_fmt<kFmtBf16>(lc, a, grid);
    if (a.fmt == kFmtInt8) return launch_fmt<kFmtInt8>(lc, a, grid);
    return cudaErrorInvalidValue;
}

}  // namespace qd
