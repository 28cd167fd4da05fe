// common.cuh - small device helpers shared by the decode kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kernels.h"

#define QD_DEV __device__ __forceinline__
#define QD_HOST_DEV_INLINE __host__ __device__ __forceinline__

namespace qd {

// ---- programmatic dependent launch ---------------------------------------
// Everything a kernel does before pdl_wait() may only touch data no earlier
// kernel of the step writes (weights, scales, tables).  pdl_launch() lets the
// next kernel's CTAs start their own weight prefetch while this one finishes.
QD_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
QD_DEV void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- global loads ----------------------------------------------------------
// Weight streams are read exactly once per step: bypass L1 allocation.
QD_DEV uint4 ld_stream(const uint4 *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ---- asynchronous global -> shared copies (per thread) -----------------------
QD_DEV void cp_async16(void *smem, const void *gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
QD_DEV void cp_async4(void *smem, const void *gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(sa), "l"(gmem) : "memory");
}
QD_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QD_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Prefetch a byte range of static data into L2 (no register or smem cost).
QD_DEV void prefetch_l2(const void *p) { asm volatile("prefetch.global.L2 [%0];" ::"l"(p)); }

QD_DEV float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

QD_DEV uint16_t float_to_bf16_bits(float f) {
    __nv_bfloat16 h = __float2bfloat16_rn(f);
    return *reinterpret_cast<uint16_t *>(&h);
}

QD_DEV uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
    // (a & b) ^ c
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6a;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

QD_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

QD_DEV half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<half2 *>(&v); }
QD_DEV uint32_t h2_as_u32(half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// ---- warp / block reductions ---------------------------------------------
QD_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

QD_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Sum over the LPR lanes of one row slot (slots are aligned groups of LPR lanes).
template <int LPR>
QD_DEV float slot_sum(float v) {
#pragma unroll
    for (int o = LPR / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---- the MLP's pending contribution to the residual ------------------------------
// k_mlp's CTAs add their partial sums of the down projection into one vector D.
// D is kept in 64-bit fixed point (units of 2^-32, |value| < 2^31) so that those
// additions are exact integer adds: the result does not depend on the order in
// which the CTAs arrive.  A partial sum is rounded once to the grid (2^-33 at
// most) and the total once back to fp32 where it is read.
QD_DEV long long delta_to_fixed(float v) { return __float2ll_rn(v * 4294967296.f); }
QD_DEV float delta_to_float(long long q) { return __ll2float_rn(q) * 2.3283064365386963e-10f; }

// ---- L2 prefetch for a later kernel -------------------------------------------
// CTA c of nc prefetches its share of each range into L2 with bulk copies of
// the TMA engine (no registers, no shared memory, nothing to wait for); the
// lines are there when a later kernel of the step streams the same bytes.
QD_DEV void l2_prefetch_share(const L2Range (&r)[kMaxL2Ranges], int c, int nc) {
    if (threadIdx.x != 0) return;
    constexpr unsigned long long kChunk = 2048;  // 16-byte units per instruction (32 KB)
#pragma unroll 1
    for (int i = 0; i < kMaxL2Ranges; ++i) {
        const char *base = static_cast<const char *>(r[i].p);
        if (!base) continue;
        const unsigned long long n = r[i].bytes / 16, per = (n + nc - 1) / nc;
        const unsigned long long lo = per * (unsigned long long)c, hi = lo + per < n ? lo + per : n;
        for (unsigned long long u = lo; u < hi; u += kChunk) {
            const unsigned sz = (unsigned)((hi - u < kChunk ? hi - u : kChunk) * 16);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(base + u * 16), "r"(sz) : "memory");
        }
    }
}

// ---- in-graph timeline (llm_timeline_steps) ---------------------------------
// When a launch carries a timestamp slot, thread 0 of every CTA raises it to
// the global timer at the CTA's exit, so the slot ends up holding the time the
// launch's last CTA finished.  Declared first in a kernel so that every return
// path records.  A null slot (the normal case) costs one predicated branch.
struct TimelineMark {
    unsigned long long *slot;
    QD_DEV ~TimelineMark() {
        if (slot && threadIdx.x == 0) {
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            atomicMax(slot, t);
        }
    }
};

}  // namespace qd
