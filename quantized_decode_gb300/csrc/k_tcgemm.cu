// k_tcgemm.cu - the prefill GEMM on the 5th-generation tensor cores:
// D[M][N] = A[M][K] * B[N][K]^T with fp16 operands and an fp32 accumulator in
// tensor memory, plus the fused epilogues of the prefill (store, residual
// add, SiLU * mul of an interleaved gate/up pair).
//
// One CTA computes one 128 x 128 output tile with 4 warps:
//   warp 0 (one lane)  TMA producer: A and B tiles of 64 K-columns into a
//                      6-stage shared-memory ring (128-byte swizzle)
//   warp 1 (one lane)  MMA issuer: 4 tcgen05.mma (K = 16 each) per stage,
//                      tcgen05.commit releases the stage when they finish
//   warp 2             allocates / frees the 128 TMEM columns
//   all 4 warps        epilogue: warp w reads TMEM lanes 32w..32w+31 (= tile
//                      rows) with tcgen05.ld and writes its rows.
// CTAs are ordered M-tile fastest, so the M-tiles that share a weight tile
// run side by side and the weight tile comes from HBM once.
//
// Every wait is bounded: on timeout the kernel records kErrTimeout, stops
// issuing, waits (bounded) for its copies in flight, frees TMEM and returns.
#include "launch_util.cuh"
#include "prefill.h"
#include "ptx.cuh"
#include "kernels.h"

namespace qd {

namespace {

constexpr int kStages = 6;
constexpr int kTileBytes = kTcBM * kTcBK * 2;  // 16 KB: an A tile and a B tile have the same shape
static_assert(kTcBM == kTcBN, "A and B tiles share one shape");

struct TcBars {
    uint64_t full[kStages], empty[kStages], done;
    uint32_t tmem;
    int abort;
    int issued;
};
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * 2 * kTileBytes + sizeof(TcBars);

QD_DEV float silu_f(float a) { return a / (1.f + __expf(-a)); }

// Epilogue of one 128 x 128 tile: warp quarter q reads TMEM lanes 32q..32q+31
// (tile rows) and writes them with the store / residual-add / SiLU*mul form.
QD_DEV void tc_epilogue(const TcGemmArgs &a, uint32_t tmem, int q, int m0, int n0, bool ok) {
    using namespace ptx;
    const int lane = threadIdx.x & 31;
    const int row = m0 + 32 * q + lane;
    const bool live = ok && row < a.M;
    const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
    if (a.mode == kEpiSwiGlu) {
#pragma unroll 1
        for (int c = 0; c < kTcBN / 2; c += 32) {
            float g[32], u[32];
            tmem_ld32(trow + c, g);
            tmem_ld32(trow + kTcBN / 2 + c, u);
            if (live) {
                uint16_t *dst = a.h + (size_t)row * a.ldh + n0 / 2 + c;
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 w;
                    w.x = h2_as_u32(__floats2half2_rn(silu_f(g[i]) * u[i], silu_f(g[i + 1]) * u[i + 1]));
                    w.y = h2_as_u32(__floats2half2_rn(silu_f(g[i + 2]) * u[i + 2], silu_f(g[i + 3]) * u[i + 3]));
                    w.z = h2_as_u32(__floats2half2_rn(silu_f(g[i + 4]) * u[i + 4], silu_f(g[i + 5]) * u[i + 5]));
                    w.w = h2_as_u32(__floats2half2_rn(silu_f(g[i + 6]) * u[i + 6], silu_f(g[i + 7]) * u[i + 7]));
                    *reinterpret_cast<uint4 *>(dst + i) = w;
                }
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < kTcBN; c += 32) {
            float v[32];
            tmem_ld32(trow + c, v);
            if (live) {
                float4 *dst = reinterpret_cast<float4 *>(a.c + (size_t)row * a.ldc + n0 + c);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    float4 o = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
                    if (a.mode == kEpiAdd) {
                        const float4 r = dst[i];
                        o.x += r.x;
                        o.y += r.y;
                        o.z += r.z;
                        o.w += r.w;
                    }
                    dst[i] = o;
                }
            }
        }
    }
}

__global__ void __launch_bounds__(128, 1)
    k_tc_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b, TcGemmArgs a) {
    using namespace ptx;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sa = base, *sb = base + kStages * kTileBytes;
    TcBars *b = reinterpret_cast<TcBars *>(base + 2 * kStages * kTileBytes);
    volatile int *abort = &b->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTcBM, n0 = blockIdx.y * kTcBN;
    const int KB = a.K / kTcBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&b->full[s], 1);
            mbar_init(&b->empty[s], 1);
        }
        mbar_init(&b->done, 1);
        b->abort = 0;
        b->issued = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tm_a);
        tma_prefetch_desc(&tm_b);
    }
    if (warp == 2) tmem_alloc(&b->tmem, kTcBN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b->tmem;

    auto fail = [&]() {
        *abort = 1;
        if (a.err) atomicCAS(a.err, kErrNone, kErrTimeout);
    };

    if (warp == 0 && lane == 0) {
        int kb = 0;
        for (; kb < KB && !*abort; ++kb) {
            const int s = kb % kStages;
            const uint32_t use = (uint32_t)(kb / kStages);
            if (!mbar_wait(&b->empty[s], (use & 1u) ^ 1u, a.wait_ns)) {
                fail();
                break;
            }
            mbar_expect_tx(&b->full[s], 2 * kTileBytes);
            tma_load_2d(sa + (size_t)s * kTileBytes, &tm_a, kb * kTcBK, m0, &b->full[s]);
            tma_load_2d(sb + (size_t)s * kTileBytes, &tm_b, kb * kTcBK, n0, &b->full[s]);
        }
        b->issued = kb;
    } else if (warp == 1 && lane == 0) {
        const uint32_t idesc = umma_idesc_f16_f32(kTcBM, kTcBN);
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % kStages;
            const uint32_t use = (uint32_t)(kb / kStages);
            if (*abort || !mbar_wait(&b->full[s], use & 1u, a.wait_ns)) {
                fail();
                break;
            }
            tc_fence_after();
            const uint32_t aa = smem_u32(sa + (size_t)s * kTileBytes), ba = smem_u32(sb + (size_t)s * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < kTcBK / 16; ++kk)
                umma_f16(tmem, umma_desc_sw128(aa + kk * 32), umma_desc_sw128(ba + kk * 32), idesc,
                         (kb | kk) != 0 ? 1u : 0u);
            umma_commit(&b->empty[s]);
        }
        // arrives once every MMA issued above has completed
        umma_commit(&b->done);
    }
    __syncwarp();

    // ---- epilogue: warp w owns tile rows 32w .. 32w + 31 ----------------------
    const bool have = mbar_wait(&b->done, 0, a.wait_ns);
    if (!have && lane == 0) fail();
    tc_fence_after();
    tc_epilogue(a, tmem, warp, m0, n0, have && !*abort);

    // ---- teardown --------------------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) {
        // copies still in flight land before the CTA's shared memory goes away
        const int issued = b->issued;
        for (int kb = issued - kStages > 0 ? issued - kStages : 0; kb < issued; ++kb)
            mbar_wait(&b->full[kb % kStages], (uint32_t)(kb / kStages) & 1u, a.wait_ns);
    }
    if (warp == 2) {
        tc_fence_after();
        tmem_free(tmem, kTcBN);
    }
}


// ---------------------------------------------------------------------------
// The prefill GEMM with the weights dequantized inside the kernel, computed
// transposed so that the weights are the tensor-memory operand:
//   D[n][m] = sum_k W[n][k] * A[m][k]   (n: 128 weight rows, m: 256 prompt rows)
// One tcgen05.mma of M = 128 (weight rows, A operand in TMEM) by N = 256
// (prompt rows, B operand in shared memory) keeps the tensor core at its full
// rate; a 128 x 128 MMA with both operands in shared memory runs at about two
// thirds of it.  The weight codes never pass through shared memory as fp16:
//   warp 0 (one lane)  TMA: the 256 x 64 activation tile and the 128 x 64
//                      code tile(s) of a k-block -> stage, `full`
//   warp 1             TMEM allocation (512 columns: the 256-column fp32
//                      accumulator and a ring of 32-column weight stages);
//                      one lane issues 4 MMAs per k-block once the converters
//                      signal `conv`, then commits `empty`
//   warps 2-9          converters: the thread for weight row t and half h
//                      turns 32 codes x scale into 16 fp16 pairs and stores
//                      them into its TMEM lane (tcgen05.st); then the
//                      epilogue: warp w reads TMEM lanes 32 (w % 4) .. for
//                      prompt columns 128 ((w - 2) / 4) .., stages the tile
//                      in shared memory, and one thread writes it with a TMA
//                      store (or a TMA fp32 add for the residual epilogue)
// Weight rows of a tile: one of up to three stacked matrices (QKV), or 64 gate
// rows then the matching 64 up rows (interleaved gate/up).
// Split K: with ksplit = 2 or 4 the CTAs of a cluster take consecutive
// k-block ranges of one tile; CTA r then owns prompt columns r T / ksplit ..
// of the result, receives the other CTAs' partial sums of those columns in its
// shared memory (distributed shared-memory stores) and adds them in rank
// order (the same sum in every run).
// ---------------------------------------------------------------------------
constexpr int kWT = 256;                         // prompt rows of a tile (the MMA's N)
constexpr int kWStages = 5;
constexpr int kWActBytes = kWT * kTcBK * 2;      // 32 KB activation tile (128-byte swizzle)
constexpr int kWCodeBytes = kTcBN * 64;          // code tile budget: 128 rows x 64 INT8 codes (INT4: half)
constexpr int kWStageBytes = kWActBytes + kWCodeBytes;
constexpr int kWACols = kTcBK / 2;               // TMEM columns of one k-block of fp16 weights
constexpr int kWTmemCols = 512;
static_assert(kWT + kWStages * kWACols <= kWTmemCols, "accumulator + weight stages fit in TMEM");
constexpr int kWMaxSplit = 4;
constexpr int kWConvWarps = 8;
constexpr int kWThreads = (2 + kWConvWarps) * 32;
constexpr int kWEpiThreads = kWConvWarps * 32;  // warps 2-9
// Epilogue staging in the (then idle) stage ring:
//   store / add     fp32 tile [256 prompt rows][128 outputs]                   128 KB
//   SwiGLU          up rows fp32 [256][64] at 0, fp16 result [256][64] after    96 KB
//   split K         receive slots [ksplit - 1][T / ksplit][128] fp32 at 0, the
//                   partial sums for the other CTAs [ksplit - 1][T / ksplit][128]
//                   at kWOutOff, then this CTA's result [T / ksplit][128] there
constexpr size_t kWSlotBytes(int ks) { return (size_t)(ks - 1) * (kWT / ks) * kTcBN * 4; }
constexpr size_t kWOutOff = (kWSlotBytes(4) > kWSlotBytes(2) ? kWSlotBytes(4) : kWSlotBytes(2)) + 1023 & ~(size_t)1023;
static_assert((size_t)kWT * kTcBN * 4 <= (size_t)kWStages * kWStageBytes, "fp32 tile fits in the ring");
static_assert((size_t)kWT * 64 * 6 <= (size_t)kWStages * kWStageBytes, "SwiGLU staging fits in the ring");
static_assert(kWOutOff + kWSlotBytes(4) <= (size_t)kWStages * kWStageBytes &&
                  kWOutOff + kWSlotBytes(2) <= (size_t)kWStages * kWStageBytes,
              "split-K slots and outgoing partial sums fit in the ring");

struct TcWBars {
    uint64_t full[kWStages], conv[kWStages], empty[kWStages], done;
    uint64_t peers_ready;  // the other CTAs of the cluster have finished their main loops
    uint64_t red_full;     // the other CTAs' partial sums of this CTA's columns have arrived
    uint32_t tmem;
    int abort;
    int issued;
};
constexpr size_t kWSmemBytes = 1024 + (size_t)kWStages * kWStageBytes + sizeof(TcWBars);

struct TcWParams {
    CUtensorMap a, w[3];
    CUtensorMap out;  // C (fp32, box 128 x T / ksplit) or H (fp16, box 64 x T)
    TcQuantB b;
    TcGemmArgs g;
    int ksplit;
};

// fp16 pair (1032 + c) of the code pair at nibble shift 0 of the half-words
QD_DEV uint32_t q_nib(uint32_t w) { return lop3_and_xor(w, 0x000F000Fu, 0x64086408u); }

__global__ void __launch_bounds__(kWThreads, 1) k_tc_gemm_q(const __grid_constant__ TcWParams P) {
    using namespace ptx;
    const TcGemmArgs &a = P.g;
    const TcQuantB &qb = P.b;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    TcWBars *b = reinterpret_cast<TcWBars *>(base + (size_t)kWStages * kWStageBytes);
    volatile int *abort = &b->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int C = P.ksplit;
    const int rank = C > 1 ? (int)cluster_rank() : 0;
    const int m0 = blockIdx.y * kWT, n0 = blockIdx.z * kTcBN;
    const int KB = a.K / kTcBK;
    const int kb0 = (int)((long long)KB * rank / C), nkb = (int)((long long)KB * (rank + 1) / C) - kb0;
    const bool int4 = qb.fmt == kFmtInt4;
    const int code_row = int4 ? 32 : 64;  // bytes of one row's codes in a k-block
    auto stage_a = [&](int s) { return base + (size_t)s * kWStageBytes; };
    auto stage_c = [&](int s) { return base + (size_t)s * kWStageBytes + kWActBytes; };
    int seg = 0, seg_row = n0;
    if (!qb.interleave)
        while (seg + 1 < qb.n_seg && seg_row >= qb.seg_rows[seg]) seg_row -= qb.seg_rows[seg++];

    if (threadIdx.x == 0) {
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&b->full[s], 1);
            mbar_init(&b->conv[s], kWConvWarps);
            mbar_init(&b->empty[s], 1);
        }
        mbar_init(&b->done, 1);
        mbar_init(&b->peers_ready, C > 1 ? C - 1 : 1);
        mbar_init(&b->red_full, C > 1 ? (C - 1) * kWEpiThreads : 1);
        tma_prefetch_desc(&P.out);
        b->abort = 0;
        b->issued = 0;
        mbar_fence_init();
        tma_prefetch_desc(&P.a);
    }
    if (warp == 1) tmem_alloc(&b->tmem, kWTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (C > 1) cluster_sync();  // every CTA's barriers exist before any remote arrive
    const uint32_t tmem = b->tmem;
    auto fail = [&]() {
        *abort = 1;
        if (a.err) atomicCAS(a.err, kErrNone, kErrTimeout);
    };

    if (warp == 0) {
        if (lane == 0) {
            pdl_launch();
            auto load_codes = [&](int s, int kb) {
                const int x = kb * code_row;
                if (qb.interleave) {
                    tma_load_2d(stage_c(s), &P.w[0], x, n0 / 2, &b->full[s]);
                    tma_load_2d(stage_c(s) + (kTcBN / 2) * code_row, &P.w[1], x, n0 / 2, &b->full[s]);
                } else {
                    tma_load_2d(stage_c(s), &P.w[seg], x, seg_row, &b->full[s]);
                }
            };
            // The first stages' weight codes depend on no earlier kernel: they go out before
            // the dependency wait (programmatic dependent launch), the activations after it.
            const int pre = nkb < kWStages ? nkb : kWStages;
            for (int i = 0; i < pre; ++i) {
                mbar_expect_tx(&b->full[i], (uint32_t)(kWActBytes + kTcBN * code_row));
                load_codes(i, kb0 + i);
            }
            pdl_wait();
            for (int i = 0; i < pre; ++i) tma_load_2d(stage_a(i), &P.a, (kb0 + i) * kTcBK, m0, &b->full[i]);
            int i = pre;
            for (; i < nkb && !*abort; ++i) {
                const int s = i % kWStages, kb = kb0 + i;
                const uint32_t use = (uint32_t)(i / kWStages);
                if (!mbar_wait(&b->empty[s], (use & 1u) ^ 1u, a.wait_ns)) {
                    fail();
                    break;
                }
                mbar_expect_tx(&b->full[s], (uint32_t)(kWActBytes + kTcBN * code_row));
                tma_load_2d(stage_a(s), &P.a, kb * kTcBK, m0, &b->full[s]);
                load_codes(s, kb);
            }
            b->issued = i;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16_f32(kTcBN, kWT);
            for (int i = 0; i < nkb; ++i) {
                const int s = i % kWStages;
                const uint32_t use = (uint32_t)(i / kWStages);
                if (*abort || !mbar_wait(&b->conv[s], use & 1u, a.wait_ns)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t ab = smem_u32(stage_a(s));
                const uint32_t wt = tmem + (uint32_t)(kWT + s * kWACols);
#pragma unroll
                for (int kk = 0; kk < kTcBK / 16; ++kk)
                    umma_f16_ts(tmem, wt + kk * 8, umma_desc_sw128(ab + kk * 32), idesc, (i | kk) != 0 ? 1u : 0u);
                umma_commit(&b->empty[s]);
            }
            umma_commit(&b->done);
        }
    } else {
        // ---- converters: warp w covers TMEM lanes 32 (w % 4) .. + 31 (= tile rows) and half
        // (w - 2) / 4 of each row's 64 codes
        const int q = warp & 3, half = (warp - 2) >> 2, t = 32 * q + lane;
        int wseg = seg, wrow = seg_row + t;
        if (qb.interleave) {
            wseg = t < kTcBN / 2 ? 0 : 1;
            wrow = n0 / 2 + (t & (kTcBN / 2 - 1));
        }
        const bool have_row = wrow < qb.seg_rows[wseg];
        const int G = a.K / kGroup;
        const uint16_t *srow = int4 && have_row ? reinterpret_cast<const uint16_t *>(qb.scale[wseg]) + (size_t)wrow * G
                                                : nullptr;
        // INT4 group scales four groups ahead in a register ring (group g in sc[g & 3])
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        const int g0 = kb0 >> 1;
        if (srow) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (g0 + j < G) sc[(g0 + j) & 3] = bf16_bits_to_float(__ldg(srow + g0 + j));
        }
        const uint32_t tdst = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(kWT + 16 * half);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % kWStages, kb = kb0 + i;
            const uint32_t use = (uint32_t)(i / kWStages);
            const bool got = __all_sync(0xffffffffu, *abort == 0 && mbar_wait(&b->full[s], use & 1u, a.wait_ns));
            if (!got) {
                if (lane == 0) fail();
                break;
            }
            uint32_t r[16];
            if (int4) {
                const int g = kb >> 1;
                const __half2 s2 = __float2half2_rn(sc[g & 3]);
                const __half2 k1032 = __floats2half2_rn(1032.f, 1032.f);
                const uint4 cw = *reinterpret_cast<const uint4 *>(stage_c(s) + (size_t)t * code_row + 16 * half);
                const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // word: codes 8c .. 8c + 7 of the k-block, pairs at nibble shifts (0,16), (4,20), (8,24), (12,28)
                    const uint32_t w = wd[j];
                    r[4 * j + 0] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w)), k1032), s2));
                    r[4 * j + 1] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w >> 4)), k1032), s2));
                    r[4 * j + 2] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w >> 8)), k1032), s2));
                    r[4 * j + 3] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w >> 12)), k1032), s2));
                }
                if ((kb & 1) && srow && g + 4 < G) sc[g & 3] = bf16_bits_to_float(__ldg(srow + g + 4));
            } else {
                // INT8: the codes themselves (exact in fp16: b ^ 0x80 = c + 128 under the exponent
                // of 1024, minus 1152); the row's fp32 scale multiplies the accumulator instead
                const uint8_t *src = stage_c(s) + (size_t)t * code_row + 32 * half;
                const __half2 k1152 = __floats2half2_rn(1152.f, 1152.f);
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const uint4 w = *reinterpret_cast<const uint4 *>(src + 16 * j);
                    const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const uint32_t x = wd[e] ^ 0x80808080u;
                        r[8 * j + 2 * e] = h2_as_u32(__hsub2(u32_as_h2(prmt(x, 0x64646464u, 0x4140u)), k1152));
                        r[8 * j + 2 * e + 1] = h2_as_u32(__hsub2(u32_as_h2(prmt(x, 0x64646464u, 0x4342u)), k1152));
                    }
                }
            }
            tmem_st16_wait(tdst + (uint32_t)(s * kWACols), r);
            // the stores are complete; order them before the MMA issuer's wait on `conv`
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b->conv[s]);
        }
    }
    __syncwarp();

    // ---- epilogue by warps 2-9: warp w reads TMEM lanes 32 (w % 4) .. + 31 (tile rows) for
    // prompt columns [128 ch, 128 ch + 128), ch = (w - 2) / 4
    if (warp >= 2) {
        const int q = warp & 3, ch = (warp - 2) >> 2, row = 32 * q + lane;
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16);
        // INT8: the fp32 scale of this lane's weight row multiplies its accumulator
        float rs = 1.f;
        if (!int4) {
            int es = seg, er = seg_row + row;
            if (qb.interleave) {
                es = row < kTcBN / 2 ? 0 : 1;
                er = n0 / 2 + (row & (kTcBN / 2 - 1));
            }
            rs = __ldg(reinterpret_cast<const float *>(qb.scale[es]) + er);
        }
        const bool issuer = warp == 2 && lane == 0;
        auto epi_sync = [] { asm volatile("bar.sync 1, %0;" ::"n"(kWEpiThreads) : "memory"); };
        const bool have = mbar_wait(&b->done, 0, a.wait_ns);
        if (!have && lane == 0) fail();
        tc_fence_after();
        // every MMA has completed, so no copy is left in flight and the ring is free
        const bool live = have && !*abort;
        if (C == 1 && a.mode == kEpiSwiGlu) {
            // gate rows (TMEM quarters 0, 1) and up rows (2, 3) of feature j meet in shared memory
            float *xu = reinterpret_cast<float *>(base);
            uint16_t *hs = reinterpret_cast<uint16_t *>(base + (size_t)kWT * 64 * 4);
            const int j = 32 * (q & 1) + lane;
            if (live && q >= 2) {
#pragma unroll 1
                for (int c = 128 * ch; c < 128 * ch + 128; c += 32) {
                    float v[32];
                    tmem_ld32(trow + c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) xu[(c + i) * 64 + j] = v[i] * rs;
                }
            }
            epi_sync();
            if (live && q < 2) {
#pragma unroll 1
                for (int c = 128 * ch; c < 128 * ch + 128; c += 32) {
                    float g[32];
                    tmem_ld32(trow + c, g);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        hs[(c + i) * 64 + j] = __half_as_ushort(__float2half_rn(silu_f(g[i] * rs) * xu[(c + i) * 64 + j]));
                }
            }
            fence_proxy_async_smem();
            epi_sync();
            if (issuer && live) {
                tma_store_2d(&P.out, hs, n0 / 2, m0);
                bulk_commit_wait_read();
            }
        } else if (C == 1) {
            float *cs = reinterpret_cast<float *>(base);  // [T][128]
            if (live) {
#pragma unroll 1
                for (int c = 128 * ch; c < 128 * ch + 128; c += 32) {
                    float v[32];
                    tmem_ld32(trow + c, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) cs[(c + i) * kTcBN + row] = v[i] * rs;
                }
            }
            fence_proxy_async_smem();
            epi_sync();
            if (issuer && live) {
                if (a.mode == kEpiAdd) tma_reduce_add_2d(&P.out, cs, n0, m0);
                else tma_store_2d(&P.out, cs, n0, m0);
                bulk_commit_wait_read();
            }
        } else {
            // split K: CTA r owns prompt columns [r W, r W + W), W = T / C; warp half ch takes
            // columns [ch W / 2, ch W / 2 + W / 2) of each W-column slice
            const int W = kWT / C, h0 = ch * (W / 2), tid = threadIdx.x - 64;
            const size_t slice = (size_t)W * kTcBN;                       // floats of one [W][128] slice
            float *slots = reinterpret_cast<float *>(base);                // [C - 1][W][128] received
            float *outs = reinterpret_cast<float *>(base + kWOutOff);      // [C - 1][W][128] to send
            auto slot_of = [](int sender, int receiver) { return sender < receiver ? sender : sender - 1; };
            // this CTA's main loop is over: its slots may be written
            if (live && issuer)
                for (int r = 0; r < C; ++r)
                    if (r != rank) mbar_arrive_cluster(cluster_map(&b->peers_ready, (uint32_t)r));
            // 1) the other CTAs' columns into local staging (row-major, as the receivers keep them)
            if (live) {
                for (int r = 0; r < C; ++r) {
                    if (r == rank) continue;
                    float *o = outs + (size_t)slot_of(r, rank) * slice;
#pragma unroll 1
                    for (int c = h0; c < h0 + W / 2; c += 32) {
                        float v[32];
                        tmem_ld32(trow + r * W + c, v);
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[(c + i) * kTcBN + row] = v[i];
                    }
                }
            }
            epi_sync();
            // 2) once every other CTA's main loop is over (its slots are free), copy with
            // consecutive threads on consecutive 16-byte words, then arrive on its `red_full`
            bool ok = live && mbar_wait_cluster(&b->peers_ready, 0, a.wait_ns);
            if (live && !ok && lane == 0) fail();
            if (ok) {
                for (int r = 0; r < C; ++r) {
                    if (r == rank) continue;
                    const float4 *src = reinterpret_cast<const float4 *>(outs + (size_t)slot_of(r, rank) * slice);
                    const uint32_t dst = cluster_map(slots + (size_t)slot_of(rank, r) * slice, (uint32_t)r);
#pragma unroll 4
                    for (int i = tid; i < (int)(slice / 4); i += kWEpiThreads) {
                        const float4 v = src[i];
                        st_cluster_v4(dst + (uint32_t)i * 16, v.x, v.y, v.z, v.w);
                    }
                    mbar_arrive_cluster(cluster_map(&b->red_full, (uint32_t)r));
                }
            }
            ok = ok && mbar_wait_cluster(&b->red_full, 0, a.wait_ns);
            if (live && !ok && lane == 0) fail();
            epi_sync();  // every thread's copies are out of `outs`, which now takes the result
            // 3) this CTA's columns: partial sums in rank order
            float *os = outs;
            if (ok) {
#pragma unroll 1
                for (int c = h0; c < h0 + W / 2; c += 32) {
                    float own[32], v[32];
                    tmem_ld32(trow + rank * W + c, own);
                    for (int r = 0; r < C; ++r) {
                        if (r == rank) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) v[i] = r == 0 ? own[i] : v[i] + own[i];
                            continue;
                        }
                        const float *p = slots + (size_t)slot_of(r, rank) * slice + (size_t)c * kTcBN + row;
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = r == 0 ? p[(size_t)i * kTcBN] : v[i] + p[(size_t)i * kTcBN];
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) os[(c + i) * kTcBN + row] = v[i] * rs;
                }
            }
            fence_proxy_async_smem();
            epi_sync();
            if (issuer && ok) {
                if (a.mode == kEpiAdd) tma_reduce_add_2d(&P.out, os, n0, m0 + rank * W);
                else tma_store_2d(&P.out, os, n0, m0 + rank * W);
                bulk_commit_wait_read();
            }
        }
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) {
        const int issued = b->issued;
        for (int i = issued - kWStages > 0 ? issued - kWStages : 0; i < issued; ++i)
            mbar_wait(&b->full[i % kWStages], (uint32_t)(i / kWStages) & 1u, a.wait_ns);
    }
    if (C > 1) cluster_sync();  // no CTA leaves while another may still write into its shared memory
    if (warp == 1) {
        tc_fence_after();
        tmem_free(tmem, kWTmemCols);
    }
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
    static EncodeFn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (EncodeFn)p;
    }
    return fn;
}

}  // namespace

cudaError_t tc_operand_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols) {
    if (!map || !base || ((uintptr_t)base & 15) || rows == 0 || cols % kTcBK) return cudaErrorInvalidValue;
    EncodeFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)kTcBM};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_tc_gemm(cudaStream_t stream, const CUtensorMap &a_map, const CUtensorMap &b_map,
                           const TcGemmArgs &a) {
    if (a.M < 1 || a.N < kTcBN || a.N % kTcBN || a.K < kTcBK || a.K % kTcBK) return cudaErrorInvalidValue;
    if (a.mode == kEpiSwiGlu ? (!a.h || a.ldh < a.N / 2 || a.ldh % 8)
                             : (!a.c || a.ldc < a.N || a.ldc % 4 || (a.mode != kEpiStore && a.mode != kEpiAdd)))
        return cudaErrorInvalidValue;
    LaunchCfg lc{};
    lc.stream = stream;
    lc.pdl = false;
    const dim3 grid((unsigned)((a.M + kTcBM - 1) / kTcBM), (unsigned)(a.N / kTcBN));
    return launch_k(lc, k_tc_gemm, grid, dim3(128), kSmemBytes, a_map, b_map, a);
}

cudaError_t tc_weight_map(CUtensorMap *map, const void *codes, int fmt, uint64_t rows, uint64_t K, int box_rows) {
    const uint64_t row_bytes = fmt == kFmtInt4 ? K / 2 : K;
    if (!map || !codes || ((uintptr_t)codes & 15) || rows == 0 || K % kTcBK || row_bytes % 16 ||
        (box_rows != kTcBN && box_rows != kTcBN / 2))
        return cudaErrorInvalidValue;
    EncodeFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(fmt == kFmtInt4 ? 32 : 64), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(codes), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t tc_act_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols) {
    if (!map || !base || ((uintptr_t)base & 15) || rows == 0 || cols % kTcBK) return cudaErrorInvalidValue;
    EncodeFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kTcBK, (cuuint32_t)kWT};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

namespace {
// Tensor map of the GEMM's output for the TMA store of the epilogue: C fp32
// [M][ldc] in boxes of 128 x box_rows, or H fp16 [M][ldh] in boxes of 64 x 256.
cudaError_t tc_out_map(CUtensorMap *map, const TcGemmArgs &a, int box_rows) {
    EncodeFn enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    const bool h = a.mode == kEpiSwiGlu;
    const void *base = h ? (const void *)a.h : (const void *)a.c;
    if ((uintptr_t)base & 15) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)(h ? a.N / 2 : a.N), (cuuint64_t)a.M};
    const cuuint64_t strides[1] = {h ? (cuuint64_t)a.ldh * 2 : (cuuint64_t)a.ldc * 4};
    const cuuint32_t box[2] = {(cuuint32_t)(h ? kTcBN / 2 : kTcBN), (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, h ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                     const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}
}  // namespace

int tc_gemm_q_split(int M, int N, int K, int mode, int n_sm) {
    const int tiles = (M + kWT - 1) / kWT * (N / kTcBN);
    int ks = 1;
    if (mode != kEpiSwiGlu)
        while (2 * ks <= kWMaxSplit && tiles * 2 * ks <= n_sm && K / kTcBK >= 2 * ks) ks *= 2;
    return ks;
}

cudaError_t launch_tc_gemm_q(cudaStream_t stream, const CUtensorMap &a_map, const CUtensorMap (&w_maps)[3],
                             const TcQuantB &b, const TcGemmArgs &a, bool pdl) {
    if (a.M < 1 || a.N < kTcBN || a.N % kTcBN || a.K < kTcBK || a.K % kTcBK) return cudaErrorInvalidValue;
    if (b.fmt != kFmtInt4 && b.fmt != kFmtInt8) return cudaErrorInvalidValue;
    if (b.fmt == kFmtInt4 && a.K % kGroup) return cudaErrorInvalidValue;
    if (b.interleave) {
        if (b.seg_rows[0] != b.seg_rows[1] || 2 * b.seg_rows[0] != a.N || !b.scale[0] || !b.scale[1])
            return cudaErrorInvalidValue;
    } else {
        int n = 0;
        if (b.n_seg < 1 || b.n_seg > 3) return cudaErrorInvalidValue;
        for (int i = 0; i < b.n_seg; ++i) {
            if (b.seg_rows[i] % kTcBN || !b.scale[i]) return cudaErrorInvalidValue;  // a tile never spans two
            n += b.seg_rows[i];
        }
        if (n != a.N) return cudaErrorInvalidValue;
    }
    if (a.mode == kEpiSwiGlu ? (!a.h || a.ldh < a.N / 2 || a.ldh % 8 || !b.interleave)
                             : (!a.c || a.ldc < a.N || a.ldc % 4 || (a.mode != kEpiStore && a.mode != kEpiAdd)))
        return cudaErrorInvalidValue;
    static int n_sm[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!n_sm[dev] && (e = cudaDeviceGetAttribute(&n_sm[dev], cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return e;
    TcWParams p;
    p.a = a_map;
    for (int i = 0; i < 3; ++i) p.w[i] = w_maps[i];
    p.b = b;
    p.g = a;
    p.ksplit = tc_gemm_q_split(a.M, a.N, a.K, a.mode, n_sm[dev]);
    if ((e = tc_out_map(&p.out, a, kWT / p.ksplit)) != cudaSuccess) return e;
    LaunchCfg lc{};
    lc.stream = stream;
    lc.pdl = pdl;
    const dim3 grid((unsigned)p.ksplit, (unsigned)((a.M + kWT - 1) / kWT), (unsigned)(a.N / kTcBN));
    return launch_kc(lc, k_tc_gemm_q, grid, dim3(kWThreads), kWSmemBytes, p.ksplit, p);
}

}  // namespace qd
