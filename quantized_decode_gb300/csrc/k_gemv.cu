// k_gemv.cu - dequant GEMVs of the decode step with fused epilogues:
//   mode 0: y = W x (+ bias)                     (single-kernel op)
//   mode 1: y += W x                             (o_proj and down: residual add)
//   mode 2: y = silu(W_gate n) * (W_up n), n = RMSNorm(x)   (fused gate/up)
// Every CTA stages the whole input vector (RMSNorm first when a gain is given)
// into shared memory as prescaled fp16 pairs, then its warps take row tiles
// round-robin and stream the weight rows with 128-bit loads.
#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kNT = 256;
constexpr int kRT = 4;

QD_DEV float silu(float a) { return a / (1.f + __expf(-a)); }

template <int FMT, int LPR>
QD_DEV void rows_dot(const void *w, const void *s, int r0, int K, int U, int j, const half2 *xs,
                     float (&out)[kRT]) {
    const size_t row_bytes = FMT == kFmtInt4 ? (size_t)K / 2 : (size_t)K;
    const uint4 *wrow[kRT];
#pragma unroll
    for (int i = 0; i < kRT; ++i)
        wrow[i] = reinterpret_cast<const uint4 *>((const char *)w + (size_t)(r0 + i) * row_bytes);
    if constexpr (FMT == kFmtInt4) {
        const uint16_t *srow[kRT];
#pragma unroll
        for (int i = 0; i < kRT; ++i) srow[i] = (const uint16_t *)s + (size_t)(r0 + i) * (K / kGroup);
        int4_tile_dots<LPR, kRT>(wrow, srow, reinterpret_cast<const uint4 *>(xs), U, j, out);
    } else {
        int8_tile_dots<LPR, kRT>(wrow, reinterpret_cast<const uint4 *>(xs), U, j, out);
#pragma unroll
        for (int i = 0; i < kRT; ++i) out[i] *= __ldg((const float *)s + r0 + i);
    }
}

// Mode 2 tiles: a slot owns kRT/2 hidden units and computes both their gate and
// up rows, so SiLU(gate)*up is formed in registers.
template <int FMT, int LPR>
QD_DEV void gateup_dot(const GemvArgs &a, int u0, int U, int j, const half2 *xs, float (&out)[kRT]) {
    constexpr int H = kRT / 2;
    const size_t row_bytes = FMT == kFmtInt4 ? (size_t)a.K / 2 : (size_t)a.K;
    const uint4 *wrow[kRT];
#pragma unroll
    for (int i = 0; i < H; ++i) {
        wrow[i] = reinterpret_cast<const uint4 *>((const char *)a.w + (size_t)(u0 + i) * row_bytes);
        wrow[H + i] = reinterpret_cast<const uint4 *>((const char *)a.w2 + (size_t)(u0 + i) * row_bytes);
    }
    if constexpr (FMT == kFmtInt4) {
        const uint16_t *srow[kRT];
#pragma unroll
        for (int i = 0; i < H; ++i) {
            srow[i] = (const uint16_t *)a.s + (size_t)(u0 + i) * (a.K / kGroup);
            srow[H + i] = (const uint16_t *)a.s2 + (size_t)(u0 + i) * (a.K / kGroup);
        }
        int4_tile_dots<LPR, kRT>(wrow, srow, reinterpret_cast<const uint4 *>(xs), U, j, out);
    } else {
        int8_tile_dots<LPR, kRT>(wrow, reinterpret_cast<const uint4 *>(xs), U, j, out);
#pragma unroll
        for (int i = 0; i < H; ++i) {
            out[i] *= __ldg((const float *)a.s + u0 + i);
            out[H + i] *= __ldg((const float *)a.s2 + u0 + i);
        }
    }
}

template <int FMT, int LPR>
__global__ void __launch_bounds__(kNT) k_gemv(GemvArgs a) {
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    constexpr int S = 32 / LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LPR, j = lane % LPR;
    const int U = FMT == kFmtInt4 ? a.K / 32 : a.K / 16;
    const int rows_per_tile = a.mode == 2 ? S * (kRT / 2) : S * kRT;
    const int n_tiles = a.N / rows_per_tile;
    const int W = gridDim.x * (kNT / 32);
    const size_t row_bytes = FMT == kFmtInt4 ? (size_t)a.K / 2 : (size_t)a.K;

    {   // warm L2 with this warp's first tile (weights only; safe before the wait)
        const int t = blockIdx.x * (kNT / 32) + warp;
        if (t < n_tiles) {
            const char *base = (const char *)a.w + (size_t)t * rows_per_tile * row_bytes;
            const size_t bytes = (size_t)rows_per_tile * row_bytes;
            for (size_t off = (size_t)lane * 128; off < bytes; off += 32 * 128) prefetch_l2(base + off);
            if (a.mode == 2) {
                const char *b2 = (const char *)a.w2 + (size_t)t * rows_per_tile * row_bytes;
                for (size_t off = (size_t)lane * 128; off < bytes; off += 32 * 128) prefetch_l2(b2 + off);
            }
        }
    }

    pdl_wait();
    half2 *xs = reinterpret_cast<half2 *>(smem);
    const float post = stage_activations<kNT>(a.x, nullptr, a.gamma, a.eps, a.K, xs, nullptr, red);
    pdl_launch();

    for (int t = blockIdx.x * (kNT / 32) + warp; t < n_tiles; t += W) {
        float out[kRT];
        if (a.mode == 2) {
            const int u0 = t * rows_per_tile + slot * (kRT / 2);
            gateup_dot<FMT, LPR>(a, u0, U, j, xs, out);
            if (j == 0) {
#pragma unroll
                for (int i = 0; i < kRT / 2; ++i)
                    a.y[u0 + i] = silu(out[i] * post) * (out[kRT / 2 + i] * post);
            }
        } else {
            const int r0 = t * rows_per_tile + slot * kRT;
            rows_dot<FMT, LPR>(a.w, a.s, r0, a.K, U, j, xs, out);
            if (j == 0) {
#pragma unroll
                for (int i = 0; i < kRT; ++i) {
                    float v = out[i] * post;
                    if (a.mode == 1) {
                        v += a.y[r0 + i];
                    } else if (a.bias) {
                        v += bf16_bits_to_float(__ldg(a.bias + r0 + i));
                    }
                    a.y[r0 + i] = v;
                }
            }
        }
    }
}

template <int FMT>
cudaError_t launch_fmt(const LaunchCfg &lc, const GemvArgs &a) {
    const int U = FMT == kFmtInt4 ? a.K / 32 : a.K / 16;
    const int lpr = pick_lpr(U);
    if (!lpr) return cudaErrorInvalidValue;
    const size_t smem = (size_t)a.K * sizeof(__half);
    const int rows_per_tile = a.mode == 2 ? (32 / lpr) * (kRT / 2) : (32 / lpr) * kRT;
    const int tiles = a.N / rows_per_tile;
    int grid = (tiles + kNT / 32 - 1) / (kNT / 32);
    if (grid > 2 * lc.n_sm) grid = 2 * lc.n_sm;
    switch (lpr) {
        case 32: return launch_k(lc, k_gemv<FMT, 32>, dim3(grid), dim3(kNT), smem, a);
        case 16: return launch_k(lc, k_gemv<FMT, 16>, dim3(grid), dim3(kNT), smem, a);
        case 8: return launch_k(lc, k_gemv<FMT, 8>, dim3(grid), dim3(kNT), smem, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool gemv_shape_ok(int fmt, int N, int K, int mode) {
    if (fmt == kFmtInt4 ? (K % 256 != 0) : (K % 128 != 0)) return false;
    const int U = fmt == kFmtInt4 ? K / 32 : K / 16;
    const int lpr = pick_lpr(U);
    if (!lpr) return false;
    const int rows_per_tile = mode == 2 ? (32 / lpr) * (kRT / 2) : (32 / lpr) * kRT;
    return N > 0 && N % rows_per_tile == 0 && (size_t)K * 2 <= 200 * 1024;
}

cudaError_t launch_gemv(const LaunchCfg &lc, int fmt, const GemvArgs &a) {
    if (fmt == kFmtInt4) return launch_fmt<kFmtInt4>(lc, a);
    if (fmt == kFmtInt8) return launch_fmt<kFmtInt8>(lc, a);
    return cudaErrorInvalidValue;
}

}  // namespace qd
