// k_lmhead.cu - final RMSNorm -> LM-head GEMV -> logits + fused greedy argmax.
//
// Each CTA stages RMSNorm(x) once, streams its row tiles through the register
// stream (bf16, or INT8 with a row scale) and keeps the running (max, lowest index) pair; the CTA's pair goes to
// a per-CTA slot, and the CTA that arrives last (arrival counter, no waiting)
// reduces the slots, writes the token and, inside the decode step, hands it to
// the next step as input and advances the position.
#include <climits>

#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

// 7 warps of 4-stage rings: measured against 16 x 3, 12 x 4, 9 x 5, 8 x 6, 6 x 8 and
// 5 x 9 on the 7B head (152064 x 3584 bf16), 7 warps were fastest by 4-40 %, and 7 x 4
// beat 7 x 6 and 7 x 7 by 2 us
constexpr int kMaxWarps = 7;
constexpr int kRT = 4;  // rows per lane
constexpr int kD = 4;   // ring depth (copies 3 steps ahead)

QD_DEV void better(float &v, int &i, float v2, int i2) {
    if (v2 > v || (v2 == v && i2 < i)) {
        v = v2;
        i = i2;
    }
}

constexpr int kLPR = kLanesPerRow;

template <int FMT>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) k_lm_head(LmHeadArgs a) {
    TimelineMark timeline_mark{a.tl};
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    __shared__ float s_val[kMaxWarps];
    __shared__ int s_idx[kMaxWarps];
    __shared__ int s_last;
    constexpr int S = 32 / kLPR;
    constexpr int TR = S * kRT;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / kLPR, j = lane % kLPR;
    const int NW = blockDim.x >> 5;
    const int gw = blockIdx.x * NW + warp, W = gridDim.x * NW;
    const int NP = slabs_per_row(FMT, a.K);
    const int U = units_per_row(FMT, a.K);
    const size_t rb = FMT == kFmtBf16 ? (size_t)a.K * 2 : (size_t)a.K;
    const size_t xbytes = ((FMT == kFmtBf16 ? (size_t)a.K * 4 : (size_t)a.K * 2) + 15) & ~(size_t)15;
    const size_t gbytes = ((size_t)a.K * 2 + 15) & ~(size_t)15;
    uint16_t *gs = reinterpret_cast<uint16_t *>((char *)smem + xbytes);  // the final norm's gain
    uint4 *ring;
    uint32_t *sring;
    warp_rings<kRT, kD>((char *)smem + xbytes + gbytes, NW, warp, ring, sring);
    float post = 1.f;
    auto sync = [&]() {
        cp_async_wait<kD - 1>();  // the gain (the ring's first steps stay in flight)
        pdl_wait();
        if constexpr (FMT == kFmtBf16)
            post = stage_activations(a.x, nullptr, a.gamma, a.eps, a.K, a.stats_in, nullptr,
                                     reinterpret_cast<float *>(smem), red, act_blk_bytes<FMT>(), gs, nullptr,
                                     nullptr, nullptr, a.x2);
        else
            post = stage_activations(a.x, nullptr, a.gamma, a.eps, a.K, a.stats_in,
                                     reinterpret_cast<half2 *>(smem), nullptr, red, act_blk_bytes<FMT>(), gs,
                                     nullptr, nullptr, nullptr, a.x2);
        pdl_launch();
    };
    auto rows = [&](int t, int i) -> RowRef {
        const int r = t * TR + slot * kRT + i;
        return {reinterpret_cast<const uint4 *>((const char *)a.w + (size_t)r * rb), nullptr};
    };
    float best = -INFINITY;
    int bidx = INT_MAX;
    auto epi = [&](int t, float(&out)[kRT]) {
        if (j != 0) return;
#pragma unroll
        for (int i = 0; i < kRT; ++i) {
            const int r = t * TR + slot * kRT + i;
            float v = out[i] * post;
            if constexpr (FMT == kFmtInt8) v *= __ldg(a.scale + r);
            a.logits[r] = v;
            better(best, bidx, v, r);
        }
    };
    gain_copy_async(a.gamma, a.K, gs);
    gemv_stream<FMT, kRT, kD>(rows, epi, sync, gw, W, a.N / TR, 0, NP, U, j, smem, ring, sring);

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
        for (int w = 1; w < NW; ++w) better(best, bidx, s_val[w], s_idx[w]);
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
    for (int c = threadIdx.x; c < (int)gridDim.x; c += blockDim.x)
        better(best, bidx, __ldcg(a.part_val + c), __ldcg(a.part_idx + c));
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
        for (int w = 1; w < NW; ++w) better(best, bidx, s_val[w], s_idx[w]);
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
    const int tiles = a.N / ((32 / kLPR) * kRT);
    int nw = (tiles + grid - 1) / grid;
    nw = nw < 2 ? 2 : (nw > kMaxWarps ? kMaxWarps : nw);  // >= 64 threads (statistics read)
    const size_t fixed = (((FMT == kFmtBf16 ? (size_t)a.K * 4 : (size_t)a.K * 2) + 15) & ~(size_t)15) +
                         (((size_t)a.K * 2 + 15) & ~(size_t)15);
    while (nw > 2 && fixed + (size_t)nw * ring_bytes_per_warp<kRT, kD>() > kMaxSmemOptin - 1024) --nw;  // wide K
    const size_t smem = fixed + (size_t)nw * ring_bytes_per_warp<kRT, kD>();
    if (smem > kMaxSmemOptin - 1024) return cudaErrorInvalidValue;
    return launch_k(lc, k_lm_head<FMT>, dim3(grid), dim3(nw * 32), smem, a);
}

}  // namespace

bool lm_head_shape_ok(int fmt, int N, int K) {
    if (fmt != kFmtBf16 && fmt != kFmtInt8) return false;
    if (K % 256 != 0 || (size_t)K * 4 > 64 * 1024) return false;
    return N > 0 && N % ((32 / kLPR) * kRT) == 0;
}

int lm_head_grid(const LaunchCfg &lc, int N) {
    const int tiles = N / kRT;
    int grid = (tiles + kMaxWarps - 1) / kMaxWarps;
    if (grid > lc.n_sm) grid = lc.n_sm;
    return grid < 1 ? 1 : grid;
}

cudaError_t launch_lm_head(const LaunchCfg &lc, const LmHeadArgs &a, int grid) {
    if (a.fmt == kFmtBf16) return launch_fmt<kFmtBf16>(lc, a, grid);
    if (a.fmt == kFmtInt8) return launch_fmt<kFmtInt8>(lc, a, grid);
    return cudaErrorInvalidValue;
}

}  // namespace qd
