// k_gemv.cu - dequant GEMVs of the decode step with fused epilogues:
//   mode 0: y = W x (+ bias)                                  (single-kernel op)
//   mode 1: y += W x                                          (o_proj and down: residual add)
//   mode 2: y = silu(W_gate n) * (W_up n), n = RMSNorm(x)      (fused gate/up)
// One CTA per SM at most.  Warps stream row tiles through lane-private
// shared-memory rings (gemv_stream); when a tile's K is split over ks warps of
// the CTA, their partial sums meet in shared memory at the end of the tile.
#include "gemv.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kMaxWarps = 16;  // 512 threads at <= 128 registers
// Ring depth: copies D - 1 steps ahead of the arithmetic.  Measured on the 7B
// INT4 decode step (in-graph times): shallow rings win -- o_proj / down at D = 2
// (down 12.1 us against 13.5 at D = 5), gate/up at D = 3 (17.0 against 17.9 at
// D = 4; D = 2 starves it, 26.7).  The fewer weight copies a kernel issues
// before its dependency wait, the sooner the input staging after the wait
// gets its round trip.  A step of INT8 (or bf16) rows covers half (a quarter)
// of the K values of an INT4 step; those keep the deeper rings (Qwen3-8B INT8
// decode was 3 % slower at the INT4 depths).
template <int FMT, int RT>
constexpr int kDepth = (FMT == kFmtInt4 || FMT == kFmtInt4A8) ? (RT >= 4 ? 3 : 2) : (RT >= 4 ? 4 : 5);

QD_DEV float silu(float a) { return a / (1.f + __expf(-a)); }

// Shared memory of the staged activations: fp16 [K], or for kFmtInt4A8 int8 [K]
// then the group scales fp32 [K/128] and the unit code sums int32 [K/32].
template <int FMT>
QD_HOST_DEV_INLINE size_t act_region_bytes(int K) {
    return FMT == kFmtInt4A8 ? (((size_t)K + 4 * (size_t)(K / 128) + 4 * (size_t)(K / 32) + 15) & ~(size_t)15)
                             : (((size_t)K * 2 + 15) & ~(size_t)15);
}
QD_HOST_DEV_INLINE size_t gain_region_bytes(int K) { return ((size_t)K * 2 + 15) & ~(size_t)15; }

// X2: the staged input is x + a.x2 (fixed point), a separate instantiation so that the
// common one keeps a compile-time null second source
template <int FMT, int RT, bool X2>
__global__ void __launch_bounds__(kMaxWarps * 32, 1) k_gemv(GemvArgs a) {
    TimelineMark timeline_mark{a.tl};
    l2_prefetch_share(a.pf, blockIdx.x, gridDim.x);
    constexpr int LPR = kLanesPerRow;
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    constexpr int S = 32 / LPR;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LPR, j = lane % LPR;
    const int NW = blockDim.x >> 5, ks = a.ks, tpc = NW / ks;
    const int kp = warp % ks, tslot = warp / ks;
    const int NP = slabs_per_row(FMT, a.K);
    const int U = units_per_row(FMT, a.K);
    const int PP = (NP + ks - 1) / ks;
    const int p_begin = kp * PP, p_end = min(NP, p_begin + PP);
    const size_t rb = int4_weights(FMT) ? (size_t)a.K / 2 : (size_t)a.K;
    const int G = a.K / kGroup;
    half2 *xs = reinterpret_cast<half2 *>(smem);
    const size_t xbytes = act_region_bytes<FMT>(a.K);
    float *a8_sx = FMT == kFmtInt4A8 ? reinterpret_cast<float *>((char *)smem + a.K) : nullptr;
    int *a8_qs = FMT == kFmtInt4A8 ? reinterpret_cast<int *>(a8_sx + a.K / kGroup) : nullptr;
    uint16_t *gs = reinterpret_cast<uint16_t *>((char *)smem + xbytes);  // the gain (when a.gamma)
    const size_t gbytes = a.gamma ? gain_region_bytes(a.K) : 0;
    uint4 *ring;
    uint32_t *sring;
    warp_rings<RT, kDepth<FMT, RT>>((char *)smem + xbytes + gbytes, NW, warp, ring, sring);
    float *kred = reinterpret_cast<float *>((char *)smem + xbytes + gbytes +
                                            (size_t)NW * ring_bytes_per_warp<RT, kDepth<FMT, RT>>()) +
                  (size_t)tslot * ks * 32 * RT;
    float post = 1.f;
    float st_ss = 0.f, st_mx = 0.f;  // statistics of what this thread writes
    const int t_first = blockIdx.x * tpc + tslot, t_stride = gridDim.x * tpc;
    // Modes 0 and 1: the epilogue inputs of the lane's first tile, loaded before
    // the dependency wait -- row scales, bias and the next norm's gain are
    // static; the residual y (mode 1) was last written two or more kernels
    // earlier, which under programmatic dependent launch has completed before
    // this kernel's CTAs are launched (each kernel signals its dependents only
    // after its own wait, i.e. after its predecessor completed).
    float pre_mul[RT], pre_add[RT], pre_g[RT];
    auto sync = [&]() {
        cp_async_wait<kDepth<FMT, RT> - 1>();  // the gain (the ring's first steps stay in flight)
        if (a.mode != 2 && j == 0 && kp == 0 && t_first < a.N / (S * RT)) {
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                const int r = t_first * S * RT + slot * RT + i;
                pre_mul[i] = FMT == kFmtInt8 ? __ldg((const float *)a.s + r) : 1.f;
                // mode 1 with fold: the MLP's pending contribution (written three kernels
                // earlier, complete by the same argument) joins the residual here
                pre_add[i] = a.mode == 1
                                 ? __ldcg(a.y + r) + (a.fold && a.fold_add ? delta_to_float(__ldcg(a.fold + r)) : 0.f)
                                 : (a.bias ? bf16_bits_to_float(__ldg(a.bias + r)) : 0.f);
                pre_g[i] = a.stats_gamma ? bf16_bits_to_float(__ldg(a.stats_gamma + r)) : 1.f;
            }
        }
        pdl_wait();
        post = stage_activations(a.x, nullptr, a.gamma, a.eps, a.K, a.stats_in, FMT == kFmtInt4A8 ? nullptr : xs,
                                 nullptr, red, act_blk_bytes<FMT>(), a.gamma ? gs : nullptr,
                                 FMT == kFmtInt4A8 ? reinterpret_cast<uint8_t *>(xs) : nullptr, a8_sx, a8_qs,
                                 X2 ? a.x2 : nullptr);
        pdl_launch();
    };
    gain_copy_async(a.gamma, a.K, gs);
    if (a.mode == 2) {
        constexpr int H = RT / 2;
        const int TU = S * H;
        auto rows = [&](int t, int i) -> RowRef {
            const int u = t * TU + slot * H + (i % H);
            const void *w = i < H ? a.w : a.w2;
            const void *s = i < H ? a.s : a.s2;
            return {reinterpret_cast<const uint4 *>((const char *)w + (size_t)u * rb),
                    (const uint16_t *)s + (size_t)u * G};
        };
        auto epi = [&](int t, float(&out)[RT]) {
            if (!ksplit_reduce<RT>(out, ks, kp, tslot, kred, j, slot, LPR) || j != 0) return;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const int u = t * TU + slot * H + i;
                float g = out[i] * post, up = out[H + i] * post;
                if constexpr (FMT == kFmtInt8) {
                    g *= __ldg((const float *)a.s + u);
                    up *= __ldg((const float *)a.s2 + u);
                }
                const float yv = silu(g) * up;
                a.y[u] = yv;
                st_ss += yv * yv;
                st_mx = fmaxf(st_mx, fabsf(yv));
            }
        };
        gemv_stream<FMT, RT, kDepth<FMT, RT>>(rows, epi, sync, t_first, t_stride, a.N / TU, p_begin, p_end, U, j, xs, ring,
                                 sring, a8_sx, a8_qs);
    } else {
        const int TR = S * RT;
        auto rows = [&](int t, int i) -> RowRef {
            const int r = t * TR + slot * RT + i;
            return {reinterpret_cast<const uint4 *>((const char *)a.w + (size_t)r * rb),
                    (const uint16_t *)a.s + (size_t)r * G};
        };
        auto epi = [&](int t, float(&out)[RT]) {
            if (!ksplit_reduce<RT>(out, ks, kp, tslot, kred, j, slot, LPR) || j != 0) return;
            const bool first = t == t_first;
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                const int r = t * TR + slot * RT + i;
                float v = out[i] * post;
                if constexpr (FMT == kFmtInt8) v *= first ? pre_mul[i] : __ldg((const float *)a.s + r);
                if (first) {
                    v += pre_add[i];
                } else if (a.mode == 1) {
                    v += __ldcg(a.y + r) + (a.fold && a.fold_add ? delta_to_float(__ldcg(a.fold + r)) : 0.f);
                } else if (a.bias) {
                    v += bf16_bits_to_float(__ldg(a.bias + r));
                }
                a.y[r] = v;
                if (a.mode == 1 && a.fold) a.fold[r] = 0;
                st_ss += v * v;
                const float gn = first ? pre_g[i] : (a.stats_gamma ? bf16_bits_to_float(__ldg(a.stats_gamma + r)) : 1.f);
                st_mx = fmaxf(st_mx, fabsf(v * gn));
            }
        };
        gemv_stream<FMT, RT, kDepth<FMT, RT>>(rows, epi, sync, t_first, t_stride, a.N / TR, p_begin, p_end, U, j, xs, ring,
                                 sring, a8_sx, a8_qs);
    }
    if (a.stats_out) write_block_stats(st_ss, st_mx, a.stats_out, red);
}

template <int FMT, int RT>
cudaError_t launch_shape(const LaunchCfg &lc, GemvArgs a, int ks) {
    constexpr int LPR = kLanesPerRow;
    const int rows_per_tile = a.mode == 2 ? (32 / LPR) * (RT / 2) : (32 / LPR) * RT;
    const int tiles = a.N / rows_per_tile;
    const size_t fixed = act_region_bytes<FMT>(a.K) + (a.gamma ? gain_region_bytes(a.K) : 0);  // activations (+ gain)
    const size_t per_warp = ring_bytes_per_warp<RT, kDepth<FMT, RT>>() + (size_t)32 * RT * 4;
    const int fit = (int)((kMaxSmemOptin - fixed) / per_warp);  // warps whose rings fit in shared memory
    GemvPlan pl = plan_gemv(tiles, ks, lc.n_sm < kStatSlots ? lc.n_sm : kStatSlots,
                            (fit < kMaxWarps ? fit : kMaxWarps) / ks * ks);
    a.ks = ks;
    const size_t smem = fixed + (size_t)pl.nw * per_warp;
    if (a.x2) {
        if constexpr (RT == 4) {
            if (a.mode != 2 || a.stats_in) return cudaErrorInvalidValue;
            return launch_k(lc, k_gemv<FMT, RT, true>, dim3(pl.grid), dim3(pl.nw * 32), smem, a);
        }
        return cudaErrorInvalidValue;
    }
    return launch_k(lc, k_gemv<FMT, RT, false>, dim3(pl.grid), dim3(pl.nw * 32), smem, a);
}

// Shape choices: K split over warps for short row counts (o_proj, down), so
// that every SM gets enough warps; 4 rows per lane for the wide gate/up.
template <int FMT>
cudaError_t launch_fmt(const LaunchCfg &lc, const GemvArgs &a) {
    const int NP = slabs_per_row(FMT, a.K);
    if (a.mode == 2) return launch_shape<FMT, 4>(lc, a, 1);
    int ks = 1;
    const int rows_per_tile = 4 * 2;  // LPR 8, RT 2
    const int tiles = a.N / rows_per_tile;
    while (ks < 4 && tiles * ks < 8 * lc.n_sm && NP / (ks * 2) >= 1) ks *= 2;
    return launch_shape<FMT, 2>(lc, a, ks);
}

}  // namespace

bool gemv_shape_ok(int fmt, int N, int K, int mode) {
    if (int4_weights(fmt) ? (K % 256 != 0) : (K % 128 != 0)) return false;
    const int rows_per_tile = mode == 2 ? 4 * 2 : 4 * 2;
    return N > 0 && N % rows_per_tile == 0 && (size_t)K * 2 <= 64 * 1024;
}

cudaError_t launch_gemv(const LaunchCfg &lc, int fmt, const GemvArgs &a) {
    if (fmt == kFmtInt4) return launch_fmt<kFmtInt4>(lc, a);
    if (fmt == kFmtInt8) return launch_fmt<kFmtInt8>(lc, a);
    if (fmt == kFmtInt4A8) return launch_fmt<kFmtInt4A8>(lc, a);
    return cudaErrorInvalidValue;
}

}  // namespace qd
