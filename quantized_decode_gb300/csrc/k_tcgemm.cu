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
// The same GEMM with the weights dequantized inside the kernel: the B operand
// arrives as INT4 (or INT8) code tiles (TMA, 128 rows x 64 codes) and four
// converter warps turn each into the fp16 128-byte-swizzled tile the MMA
// reads (two threads per weight row, half of its 64 codes each: code x scale
// is exact in fp16 for INT4; INT8 rounds once), so no fp16 copy of the
// weights goes through HBM.
//   warp 0 (one lane)  TMA: A tile and code tile(s) -> stage, `full`
//   warp 1             TMEM allocation; one lane issues the MMAs once the
//                      converters signal `conv`, commits `empty`
//   warps 2-9          converters; warps 2-5 then run the epilogue (warp w:
//                      TMEM lanes 32 (w % 4) .. +31)
// Weight rows of a 128-row tile: one of up to three stacked matrices (QKV),
// or 64 gate rows then the matching 64 up rows (interleaved gate/up).
// ---------------------------------------------------------------------------
constexpr int kQStages = 5;
constexpr int kQCodeBytes = kTcBN * 64;  // code tile budget: 128 rows x 64 INT8 codes (INT4 uses half)
constexpr int kQStageBytes = 2 * kTileBytes + kQCodeBytes;

struct TcQBars {
    uint64_t full[kQStages], conv[kQStages], empty[kQStages], done;
    uint32_t tmem;
    int abort;
    int issued;
};
constexpr size_t kQSmemBytes = 1024 + (size_t)kQStages * kQStageBytes + sizeof(TcQBars);
constexpr int kQConvWarps = 8;
constexpr int kQThreads = (2 + kQConvWarps) * 32;

struct TcQParams {
    CUtensorMap a, w[3];
    TcQuantB b;
    TcGemmArgs g;
};

// fp16 pair (1032 + c) of the code pair at nibble shift 0 of the half-words
QD_DEV uint32_t q_nib(uint32_t w) { return lop3_and_xor(w, 0x000F000Fu, 0x64086408u); }

__global__ void __launch_bounds__(kQThreads, 1) k_tc_gemm_q(const __grid_constant__ TcQParams P) {
    using namespace ptx;
    const TcGemmArgs &a = P.g;
    const TcQuantB &qb = P.b;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    TcQBars *b = reinterpret_cast<TcQBars *>(base + (size_t)kQStages * kQStageBytes);
    volatile int *abort = &b->abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * kTcBM, n0 = blockIdx.y * kTcBN;
    const int KB = a.K / kTcBK;
    const bool int4 = qb.fmt == kFmtInt4;
    const int code_row = int4 ? 32 : 64;  // bytes of one row's codes in a k-block
    auto stage_a = [&](int s) { return base + (size_t)s * kQStageBytes; };
    auto stage_b = [&](int s) { return base + (size_t)s * kQStageBytes + kTileBytes; };
    auto stage_c = [&](int s) { return base + (size_t)s * kQStageBytes + 2 * kTileBytes; };
    // weight rows of this tile: segment and first row (stacked), or the pair base (interleaved)
    int seg = 0, seg_row = n0;
    if (!qb.interleave)
        while (seg + 1 < qb.n_seg && seg_row >= qb.seg_rows[seg]) seg_row -= qb.seg_rows[seg++];

    if (threadIdx.x == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(&b->full[s], 1);
            mbar_init(&b->conv[s], kQConvWarps);
            mbar_init(&b->empty[s], 1);
        }
        mbar_init(&b->done, 1);
        b->abort = 0;
        b->issued = 0;
        mbar_fence_init();
        tma_prefetch_desc(&P.a);
    }
    if (warp == 1) tmem_alloc(&b->tmem, kTcBN);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = b->tmem;
    auto fail = [&]() {
        *abort = 1;
        if (a.err) atomicCAS(a.err, kErrNone, kErrTimeout);
    };

    if (warp == 0) {
        if (lane == 0) {
            int kb = 0;
            for (; kb < KB && !*abort; ++kb) {
                const int s = kb % kQStages;
                const uint32_t use = (uint32_t)(kb / kQStages);
                if (!mbar_wait(&b->empty[s], (use & 1u) ^ 1u, a.wait_ns)) {
                    fail();
                    break;
                }
                mbar_expect_tx(&b->full[s], (uint32_t)(kTileBytes + kTcBN * code_row));
                tma_load_2d(stage_a(s), &P.a, kb * kTcBK, m0, &b->full[s]);
                const int x = kb * code_row;
                if (qb.interleave) {
                    tma_load_2d(stage_c(s), &P.w[0], x, n0 / 2, &b->full[s]);
                    tma_load_2d(stage_c(s) + (kTcBN / 2) * code_row, &P.w[1], x, n0 / 2, &b->full[s]);
                } else {
                    tma_load_2d(stage_c(s), &P.w[seg], x, seg_row, &b->full[s]);
                }
            }
            b->issued = kb;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = umma_idesc_f16_f32(kTcBM, kTcBN);
            for (int kb = 0; kb < KB; ++kb) {
                const int s = kb % kQStages;
                const uint32_t use = (uint32_t)(kb / kQStages);
                if (*abort || !mbar_wait(&b->conv[s], use & 1u, a.wait_ns)) {
                    fail();
                    break;
                }
                tc_fence_after();
                const uint32_t aa = smem_u32(stage_a(s)), ba = smem_u32(stage_b(s));
#pragma unroll
                for (int kk = 0; kk < kTcBK / 16; ++kk)
                    umma_f16(tmem, umma_desc_sw128(aa + kk * 32), umma_desc_sw128(ba + kk * 32), idesc,
                             (kb | kk) != 0 ? 1u : 0u);
                umma_commit(&b->empty[s]);
            }
            umma_commit(&b->done);
        }
    } else {
        // ---- converters: threads t and t + 128 share weight row t of the tile
        const int ct = threadIdx.x - 64, t = ct & (kTcBN - 1), half = ct >> 7;
        int wseg = seg, wrow = seg_row + t;
        if (qb.interleave) {
            wseg = t < kTcBN / 2 ? 0 : 1;
            wrow = n0 / 2 + (t & (kTcBN / 2 - 1));
        }
        const bool have_row = wrow < (qb.interleave ? qb.seg_rows[wseg] : qb.seg_rows[wseg]);
        const int G = a.K / kGroup;
        const uint16_t *srow = int4 && have_row ? reinterpret_cast<const uint16_t *>(qb.scale[wseg]) + (size_t)wrow * G
                                                : nullptr;
        float sc8 = 0.f;
        if (!int4 && have_row) sc8 = __ldg(reinterpret_cast<const float *>(qb.scale[wseg]) + wrow);
        // INT4 group scales four groups ahead in a register ring (group g in sc[g & 3])
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        if (srow) {
#pragma unroll
            for (int g = 0; g < 4; ++g)
                if (g < G) sc[g] = bf16_bits_to_float(__ldg(srow + g));
        }
        for (int kb = 0; kb < KB; ++kb) {
            const int s = kb % kQStages;
            const uint32_t use = (uint32_t)(kb / kQStages);
            const bool got = __all_sync(0xffffffffu, *abort == 0 && mbar_wait(&b->full[s], use & 1u, a.wait_ns));
            if (!got) {
                if (lane == 0) fail();
                break;
            }
            const uint8_t *src = stage_c(s) + (size_t)t * code_row;
            uint8_t *dst = stage_b(s) + (size_t)t * 128;
            if (int4) {
                const int g = kb >> 1;
                const __half2 s2 = __float2half2_rn(sc[g & 3]);
                const __half2 k1032 = __floats2half2_rn(1032.f, 1032.f);
                const uint4 cw = *reinterpret_cast<const uint4 *>(src + 16 * half);
                const uint32_t wd[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    // word c: codes 8c .. 8c + 7 of the k-block, lanes at shifts 0,16,4,20,8,24,12,28
                    const int c = 4 * half + q;
                    const uint32_t w = wd[q];
                    uint4 o;
                    o.x = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w)), k1032), s2));
                    o.y = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w >> 4)), k1032), s2));
                    o.z = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w >> 8)), k1032), s2));
                    o.w = h2_as_u32(__hmul2(__hsub2(u32_as_h2(q_nib(w >> 12)), k1032), s2));
                    *reinterpret_cast<uint4 *>(dst + ((c ^ (t & 7)) << 4)) = o;
                }
                if ((kb & 1) && srow && g + 4 < G) sc[g & 3] = bf16_bits_to_float(__ldg(srow + g + 4));
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int c = 4 * half + q;
                    const uint2 w = *reinterpret_cast<const uint2 *>(src + 8 * c);
                    uint4 o;
                    o.x = h2_as_u32(__floats2half2_rn((float)(int8_t)(w.x & 0xFF) * sc8, (float)(int8_t)((w.x >> 8) & 0xFF) * sc8));
                    o.y = h2_as_u32(__floats2half2_rn((float)(int8_t)((w.x >> 16) & 0xFF) * sc8, (float)(int8_t)(w.x >> 24) * sc8));
                    o.z = h2_as_u32(__floats2half2_rn((float)(int8_t)(w.y & 0xFF) * sc8, (float)(int8_t)((w.y >> 8) & 0xFF) * sc8));
                    o.w = h2_as_u32(__floats2half2_rn((float)(int8_t)((w.y >> 16) & 0xFF) * sc8, (float)(int8_t)(w.y >> 24) * sc8));
                    *reinterpret_cast<uint4 *>(dst + ((c ^ (t & 7)) << 4)) = o;
                }
            }
            // generic-proxy writes -> visible to the tensor core (async proxy) before the signal
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&b->conv[s]);
        }
    }
    __syncwarp();

    // ---- epilogue by converter warps 2-5 (one per TMEM lane quarter)
    if (warp >= 2 && warp < 6) {
        const bool have = mbar_wait(&b->done, 0, a.wait_ns);
        if (!have && lane == 0) fail();
        tc_fence_after();
        tc_epilogue(a, tmem, warp & 3, m0, n0, have && !*abort);
    }

    // ---- teardown
    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort) {
        const int issued = b->issued;
        for (int kb = issued - kQStages > 0 ? issued - kQStages : 0; kb < issued; ++kb)
            mbar_wait(&b->full[kb % kQStages], (uint32_t)(kb / kQStages) & 1u, a.wait_ns);
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_free(tmem, kTcBN);
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

cudaError_t launch_tc_gemm_q(cudaStream_t stream, const CUtensorMap &a_map, const CUtensorMap (&w_maps)[3],
                             const TcQuantB &b, const TcGemmArgs &a) {
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
    if (a.mode == kEpiSwiGlu ? (!a.h || a.ldh < a.N / 2 || a.ldh % 8)
                             : (!a.c || a.ldc < a.N || a.ldc % 4 || (a.mode != kEpiStore && a.mode != kEpiAdd)))
        return cudaErrorInvalidValue;
    TcQParams p;
    p.a = a_map;
    for (int i = 0; i < 3; ++i) p.w[i] = w_maps[i];
    p.b = b;
    p.g = a;
    LaunchCfg lc{};
    lc.stream = stream;
    lc.pdl = false;
    const dim3 grid((unsigned)((a.M + kTcBM - 1) / kTcBM), (unsigned)(a.N / kTcBN));
    return launch_k(lc, k_tc_gemm_q, grid, dim3(kQThreads), kQSmemBytes, p);
}

}  // namespace qd
