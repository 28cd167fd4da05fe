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
#include "step.h"  // kErrTimeout

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
    const int row = m0 + 32 * warp + lane;
    const bool live = have && row < a.M && !*abort;
    const uint32_t trow = tmem + ((uint32_t)(32 * warp) << 16);
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

}  // namespace qd
