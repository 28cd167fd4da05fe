// k_mlp.cu - the decode step's MLP block as one kernel.
//
// CTA c owns a slice [f0, f1) of the MLP's hidden units and computes
//   phase 1:  u_f = silu(W_gate[f] . n) * (W_up[f] . n)      f in [f0, f1),  n = RMSNorm(x)
//   phase 2:  D  += W_down[:, f0:f1] u[f0:f1]                 (all h rows; integer reductions in L2)
// ("从头开始手写一个Qwen的Naive CUDA Kernel推理引擎(一)", "SwiGLU"; the down
// projection of "How To Construct Your Personal LLM Runtime From Scratch", §3).
// The down projection of a slice starts inside the CTA that produced the slice,
// so the block needs no grid-wide hand-off between gate/up and down and streams
// its 3 * F * h weights as one kernel.  D is the MLP's contribution to the
// residual: it is zero when the kernel starts and the next o_proj folds it into x
// (and zeroes it), while the next QKV and the LM head read x + D.  The partial
// sums of different CTAs meet in D through integer red.add in 64-bit fixed point
// (delta_to_fixed), so the result does not depend on the order the CTAs arrive.
//
// Phase 1 is the gate/up GEMV of k_gemv.cu (lane-private cp.async rings) run over
// the CTA's rows only.  Phase 2 reads W_down as the engine repacks it at create
// time: unit-major [F / C][h][16 bytes] (C = 32 INT4 or 16 INT8 codes per 16
// bytes), so a CTA's units are one contiguous block that it prefetches into L2
// at its start, and INT4 scales as [F / 128][h].
#include "gemv.cuh"
#include "launch_util.cuh"
#include "ptx.cuh"

namespace qd {

namespace {

constexpr int kNW = 8;       // warps per CTA (RT = 4 rings, 128 registers in phase 1)
constexpr int kRT = 4;       // rows per lane in phase 1: 2 gate + 2 up
constexpr int kD = 4;        // ring depth of phase 1
constexpr int kMaxRows = 16;   // rows per thread in phase 2 (h <= 16 * 256)
constexpr int kMaxCols = 512;  // hidden units per CTA (u slice in shared memory)
constexpr size_t kMaxUnitBytes = 4096 * 16;  // one unit of every down row, h <= 4096
constexpr uint32_t kBulkPiece = 16384;        // bytes per bulk copy instruction

// Bulk copy (TMA engine) of n bytes global -> shared, completion counted on bar.
QD_DEV void bulk_g2s(void *dst, const void *src, uint32_t n, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            ptx::smem_u32(dst)),
        "l"(src), "r"(n), "r"(ptx::smem_u32(bar))
        : "memory");
}

QD_DEV float silu(float a) { return a / (1.f + __expf(-a)); }

template <int FMT>
constexpr int cols_per_unit() { return FMT == kFmtInt4 ? 32 : 16; }

// The CTA's units [u0, u1) of NU, as even as the grid allows.
QD_HOST_DEV_INLINE void unit_span(int NU, int c, int G, int &u0, int &u1) {
    u0 = (int)((long long)NU * c / G);
    u1 = (int)((long long)NU * (c + 1) / G);
}

template <int FMT>
QD_DEV float unit_dot(uint4 q, const uint4 (&x)[4]) {
    if constexpr (FMT == kFmtInt4) {
        return int4_unit_dot(q, x);
    } else {
        const uint4 x2[2] = {x[0], x[1]};
        return int8_unit_dot(q, x2);
    }
}

template <int FMT>
__global__ void __launch_bounds__(kNW * 32, 1) k_mlp(MlpArgs a) {
    TimelineMark timeline_mark{a.tl};
    constexpr int LPR = kLanesPerRow;
    constexpr int S = 32 / LPR;
    constexpr int H = kRT / 2;
    constexpr int TU = S * H;               // hidden units per phase-1 tile
    constexpr int CU = cols_per_unit<FMT>();
    extern __shared__ uint4 smem[];
    __shared__ float red[64];
    __shared__ float us[kMaxCols];          // u of the CTA's slice (fp32)
    __shared__ __align__(16) __half us16[kMaxCols];  // u * 2^-e as fp16 (phase 2 activations)
    __shared__ float s_post2;

    const int K = a.h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int slot = lane / LPR, j = lane % LPR;
    const int NU = a.F / CU;
    int u0, u1;
    unit_span(NU, blockIdx.x, gridDim.x, u0, u1);
    const int nu = u1 - u0, f0 = u0 * CU, ncol = nu * CU;
    const size_t unit_bytes = (size_t)a.h * 16;  // one unit of every down row

    // Phase 2's weights do not depend on anything: start their way into L2 now.
    if (threadIdx.x == 0 && a.prefetch_down && nu > 0) {
        L2Range r[kMaxL2Ranges] = {};
        r[0] = {reinterpret_cast<const char *>(a.wd) + (size_t)u0 * unit_bytes, (unsigned long long)nu * unit_bytes};
        if constexpr (FMT == kFmtInt4) {
            const int g0 = u0 / 4, g1 = (u1 + 3) / 4;
            r[1] = {static_cast<const uint16_t *>(a.sd) + (size_t)g0 * a.h, (unsigned long long)(g1 - g0) * a.h * 2};
        }
        l2_prefetch_share(r, 0, 1);
    }

    const int NP = slabs_per_row(FMT, K);
    const int U = units_per_row(FMT, K);
    const size_t rb = FMT == kFmtInt4 ? (size_t)K / 2 : (size_t)K;
    const int G = K / kGroup;
    half2 *xs = reinterpret_cast<half2 *>(smem);
    const size_t xbytes = ((size_t)K * 2 + 15) & ~(size_t)15;
    uint16_t *gs = reinterpret_cast<uint16_t *>((char *)smem + xbytes);
    const size_t gbytes = ((size_t)K * 2 + 15) & ~(size_t)15;
    uint4 *ring;
    uint32_t *sring;
    warp_rings<kRT, kD>((char *)smem + xbytes + gbytes, kNW, warp, ring, sring);
    // phase 2's three unit buffers: its own region after the rings, then two in the rings
    uint4 *bufs[3];
    bufs[0] = reinterpret_cast<uint4 *>((char *)smem + xbytes + gbytes + (size_t)kNW * ring_bytes_per_warp<kRT, kD>());
    bufs[1] = reinterpret_cast<uint4 *>((char *)smem + xbytes + gbytes);
    bufs[2] = reinterpret_cast<uint4 *>((char *)smem + xbytes + gbytes + kMaxUnitBytes);
    __shared__ __align__(8) uint64_t bar[3];
    if (threadIdx.x == 0) {
#pragma unroll
        for (int i = 0; i < 3; ++i) ptx::mbar_init(&bar[i], 1);
        ptx::mbar_fence_init();
    }
    __syncthreads();
    // the first unit does not depend on anything either: on its way now
    auto issue0 = [&]() {
        const uint32_t ublk = (uint32_t)unit_bytes;
        const char *src = reinterpret_cast<const char *>(a.wd) + (size_t)u0 * unit_bytes;
        ptx::mbar_expect_tx(&bar[0], ublk);
        for (uint32_t off = 0; off < ublk; off += kBulkPiece) {
            const uint32_t n = ublk - off < kBulkPiece ? ublk - off : kBulkPiece;
            bulk_g2s(reinterpret_cast<char *>(bufs[0]) + off, src + off, n, &bar[0]);
        }
    };
    if (threadIdx.x == 0 && nu > 0) issue0();
    float post = 1.f;
    auto sync = [&]() {
        cp_async_wait<kD - 1>();  // the gain (the ring's first steps stay in flight)
        pdl_wait();
        post = stage_activations(a.x, nullptr, a.gamma, a.eps, K, a.stats_in, xs, nullptr, red,
                                 act_blk_bytes<FMT>(), gs);
        pdl_launch();
    };
    gain_copy_async(a.gamma, K, gs);

    // ---- phase 1: the gate/up rows of the slice
    auto rows = [&](int t, int i) -> RowRef {
        const int f = f0 + t * TU + slot * H + (i % H);
        const void *w = i < H ? a.wg : a.wu;
        const void *s = i < H ? a.sg : a.su;
        return {reinterpret_cast<const uint4 *>((const char *)w + (size_t)f * rb), (const uint16_t *)s + (size_t)f * G};
    };
    auto epi = [&](int t, float(&out)[kRT]) {
        if (j != 0) return;
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const int lf = t * TU + slot * H + i;
            float g = out[i] * post, up = out[H + i] * post;
            if constexpr (FMT == kFmtInt8) {
                g *= __ldg((const float *)a.sg + f0 + lf);
                up *= __ldg((const float *)a.su + f0 + lf);
            }
            us[lf] = silu(g) * up;
        }
    };
    gemv_stream<FMT, kRT, kD>(rows, epi, sync, warp, kNW, ncol / TU, 0, NP, U, j, xs, ring, sring);
    __syncthreads();

    // ---- the slice as fp16 activations, scaled by 2^-e so that |u| * 2^-e <= 1
    if (warp == 0) {
        float m = 0.f;
        for (int i = lane; i < ncol; i += 32) m = fmaxf(m, fabsf(us[i]));
        m = warp_max(m);
        int e = 0;
        if (m > 0.f) frexpf(m, &e);
        const float pre = ldexpf(1.f, -e);
        for (int i = lane; i < ncol; i += 32) us16[i] = __float2half_rn(us[i] * pre);
        if (lane == 0) s_post2 = ldexpf(1.f, e);
    }
    __syncthreads();
    const float post2 = s_post2;

    // ---- phase 2: D[r] += sum over the slice's units of W_down[r][unit] . u[unit]
    // A unit of the slice is one contiguous block of the repacked W_down (16 bytes of
    // every row).  Blocks reach shared memory by TMA bulk copies into three buffers:
    // the first into its own region, issued at the kernel's start; the others into
    // phase 1's rings, free once phase 1 is done.  Thread t multiplies rows t + 256 i
    // of each block against that unit's activations and keeps the row sums.
    constexpr int XC = FMT == kFmtInt4 ? 4 : 2;  // 16-byte activation chunks per unit
    float acc[kMaxRows];
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) acc[i] = 0.f;
    const uint32_t ublk = (uint32_t)unit_bytes;
    int uses[3] = {nu > 0 ? 1 : 0, 0, 0};  // thread 0: copies issued into each buffer
    auto issue = [&](int k) {  // thread 0: unit k of the slice into buffer k % 3
        uint4 *dst = bufs[k % 3];
        const char *src = reinterpret_cast<const char *>(a.wd) + (size_t)(u0 + k) * unit_bytes;
        ++uses[k % 3];
        // the block's earlier generic accesses of the buffer (ordered before this
        // thread by the preceding barrier) come before the copy's writes
        ptx::fence_proxy_async_smem();
        ptx::mbar_expect_tx(&bar[k % 3], ublk);
        for (uint32_t off = 0; off < ublk; off += kBulkPiece) {
            const uint32_t n = ublk - off < kBulkPiece ? ublk - off : kBulkPiece;
            bulk_g2s(reinterpret_cast<char *>(dst) + off, src + off, n, &bar[k % 3]);
        }
    };
    if (threadIdx.x == 0) {
        if (nu > 1) issue(1);
        if (nu > 2) issue(2);
    }
    // INT4: the scales of this thread's rows for the (at most 3) groups the slice's
    // units fall in, loaded now so that their latency is off the unit loop
    const int gbase = u0 >> 2;
    float sc[3][kMaxRows];
    if constexpr (FMT == kFmtInt4) {
        const uint16_t *sd = static_cast<const uint16_t *>(a.sd);
        const int ng = ((u1 - 1) >> 2) - gbase + 1;
#pragma unroll
        for (int g = 0; g < 3; ++g)
#pragma unroll
            for (int i = 0; i < kMaxRows; ++i) {
                const int r = threadIdx.x + kNW * 32 * i;
                sc[g][i] = g < ng && r < a.h ? bf16_bits_to_float(__ldg(sd + (size_t)(gbase + g) * a.h + r)) : 0.f;
            }
    }
    bool ok = true;
#pragma unroll 1
    for (int k = 0; k < nu; ++k) {
        const uint32_t par = (uint32_t)(k / 3) & 1u;
        // bounded wait; the block decides together whether to go on
        if (__syncthreads_or(!ptx::mbar_wait(&bar[k % 3], par, a.wait_ns))) {
            ok = false;
            if (threadIdx.x == 0 && a.err) atomicCAS(a.err, kErrNone, kErrTimeout);
            break;
        }
        uint4 xr[4];
        const uint4 *x4 = reinterpret_cast<const uint4 *>(us16 + k * CU);
#pragma unroll
        for (int c = 0; c < 4; ++c) xr[c] = c < XC ? x4[c] : make_uint4(0u, 0u, 0u, 0u);
        const uint4 *blk = bufs[k % 3];
        const int gi = ((u0 + k) >> 2) - gbase;
#pragma unroll
        for (int i = 0; i < kMaxRows; ++i) {
            const int r = threadIdx.x + kNW * 32 * i;
            if (r < a.h) {
                const float d = unit_dot<FMT>(blk[r], xr);
                if constexpr (FMT == kFmtInt4) {
                    acc[i] = fmaf(d, gi == 0 ? sc[0][i] : (gi == 1 ? sc[1][i] : sc[2][i]), acc[i]);
                } else {
                    acc[i] += d;
                }
            }
        }
        __syncthreads();  // every thread is done with the buffer before it is refilled
        if (threadIdx.x == 0 && k + 3 < nu) issue(k + 3);
    }
    if (!ok) {
        // a copy did not land within the bound: wait (bounded) for the last copy
        // issued into each buffer (copies into a buffer complete in order), then
        // leave without touching D
        if (threadIdx.x == 0)
            for (int b = 0; b < 3; ++b)
                if (uses[b] > 0) ptx::mbar_wait(&bar[b], (uint32_t)(uses[b] - 1) & 1u, a.wait_ns);
        return;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kMaxRows; ++i) {
        const int r = threadIdx.x + kNW * 32 * i;
        if (r < a.h && nu > 0) {
            float v = acc[i] * post2;
            if constexpr (FMT == kFmtInt8) v *= __ldg(static_cast<const float *>(a.sd) + r);
            // exact integer add: the total does not depend on the CTAs' order
            atomicAdd(reinterpret_cast<unsigned long long *>(a.D) + r, (unsigned long long)delta_to_fixed(v));
        }
    }
    __syncthreads();
}

// W_down [h][F] (row-major; INT4 ValueShuffle words or INT8 codes) ->
// unit-major [F / C][h][16 B]; INT4 scales [h][F / 128] -> [F / 128][h].
__global__ void k_repack_down(const uint4 *__restrict__ w, uint4 *__restrict__ out, int h, int units_per_row,
                              const uint16_t *__restrict__ s, uint16_t *__restrict__ s_out, int groups) {
    const size_t n = (size_t)h * units_per_row;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / units_per_row, u = i % units_per_row;
        out[u * h + r] = w[i];
    }
    if (s) {
        const size_t ng = (size_t)h * groups;
        for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < ng; i += (size_t)gridDim.x * blockDim.x) {
            const size_t r = i / groups, g = i % groups;
            s_out[g * h + r] = s[i];
        }
    }
}

template <int FMT>
size_t mlp_smem(int h) {
    const size_t x = ((size_t)h * 2 + 15) & ~(size_t)15;
    static_assert(kNW * ring_bytes_per_warp<kRT, kD>() >= 2 * kMaxUnitBytes, "two unit buffers in the rings");
    return 2 * x + (size_t)kNW * ring_bytes_per_warp<kRT, kD>() + (size_t)h * 16;
}

}  // namespace

bool mlp_shape_ok(int fmt, int h, int F) {
    if (fmt != kFmtInt4 && fmt != kFmtInt8) return false;
    const int cu = fmt == kFmtInt4 ? 32 : 16;
    if (h % 256 != 0 || h > kMaxRows * kNW * 32 || F % cu != 0) return false;
    if (fmt == kFmtInt4 && F % kGroup != 0) return false;
    const size_t smem = fmt == kFmtInt4 ? mlp_smem<kFmtInt4>(h) : mlp_smem<kFmtInt8>(h);
    return smem + 4096 <= kMaxSmemOptin;
}

int mlp_grid(const LaunchCfg &lc, int fmt, int F) {
    const int NU = F / (fmt == kFmtInt4 ? 32 : 16);
    int g = lc.n_sm < NU ? lc.n_sm : NU;
    // every CTA's slice fits the shared u buffer
    const int cu = fmt == kFmtInt4 ? 32 : 16;
    while ((NU + g - 1) / g > 8) ++g;  // phase 2 takes at most 8 units per CTA
    return g;
}

cudaError_t launch_mlp(const LaunchCfg &lc, int fmt, const MlpArgs &a) {
    if (!mlp_shape_ok(fmt, a.h, a.F) || !a.D) return cudaErrorInvalidValue;
    const int grid = mlp_grid(lc, fmt, a.F);
    if (fmt == kFmtInt4)
        return launch_k(lc, k_mlp<kFmtInt4>, dim3(grid), dim3(kNW * 32), mlp_smem<kFmtInt4>(a.h), a);
    return launch_k(lc, k_mlp<kFmtInt8>, dim3(grid), dim3(kNW * 32), mlp_smem<kFmtInt8>(a.h), a);
}

cudaError_t mlp_repack_down(int fmt, const void *w, const void *s, int h, int F, void *w_out, void *s_out,
                            cudaStream_t stream) {
    const int upr = fmt == kFmtInt4 ? F / 32 : F / 16;
    const int groups = fmt == kFmtInt4 ? F / kGroup : 0;
    k_repack_down<<<1024, 256, 0, stream>>>(static_cast<const uint4 *>(w), static_cast<uint4 *>(w_out), h, upr,
                                            fmt == kFmtInt4 ? static_cast<const uint16_t *>(s) : nullptr,
                                            static_cast<uint16_t *>(s_out), groups);
    return cudaGetLastError();
}

}  // namespace qd
