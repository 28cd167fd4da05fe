// k_prefill.cu - the non-GEMM kernels of the prompt (prefill) pass:
//   k_dequant    INT4 / INT8 weight rows -> fp16 rows (GEMM B operand)
//   k_embed      token rows of the bf16 embedding -> fp32 residual rows
//   k_rmsnorm    fp32 residual rows -> RMSNorm * gain -> fp16 (GEMM A operand)
//   k_qkv_rows   bias, per-head q/k RMSNorm, RoPE, K/V -> bf16 pages, q -> bf16 hi/lo
//   k_attn_rows  causal GQA flash attention over the paged cache (mma.sync)
//
// fp16 holds every INT4 weight exactly: a code has at most 3 significant bits
// and a bf16 scale 8, and 11 fit fp16's significand (scales above 2^-14 stay
// normal).  INT8 weights dequantized to fp16 (7 + 24 bits) round once; the
// prefill GEMM instead keeps INT8 codes exact and scales each row's fp32 sum.
#include "common.cuh"
#include "launch_util.cuh"
#include "prefill.h"

namespace qd {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// Dequantization.  One thread per 8 codes (one 32-bit INT4 word / 8 INT8
// bytes) -> one 16-byte fp16 store.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_dequant(DequantArgs a) {
    const int rows_out = a.w2 ? 2 * a.N : a.N;
    const int wpr = a.K / 8;  // 8-code units per row
    const long long total = (long long)rows_out * wpr;
    for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < total;
         u += (long long)gridDim.x * blockDim.x) {
        const int r = (int)(u / wpr), c8 = (int)(u % wpr);
        int src = r;
        const void *w = a.w, *s = a.s;
        if (a.w2) {
            const int t = r / 128, i = r % 128;
            src = 64 * t + (i & 63);
            if (i >= 64) {
                w = a.w2;
                s = a.s2;
            }
        }
        float v[8];
        if (a.fmt == kFmtInt4) {
            const uint32_t word = __ldg(reinterpret_cast<const uint32_t *>(w) + (size_t)src * wpr + c8);
            const float sc = bf16_bits_to_float(__ldg(reinterpret_cast<const uint16_t *>(s) +
                                                      (size_t)src * (a.K / kGroup) + (c8 * 8) / kGroup));
            // lane i of the octet sits at bit shift 0,16,4,20,8,24,12,28
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int sh = ((i & 1) << 4) | ((i >> 1) << 2);
                const int code = ((int)((word >> sh) & 0xFu) ^ 8) - 8;
                v[i] = (float)code * sc;
            }
        } else {
            const uint2 b = __ldg(reinterpret_cast<const uint2 *>(reinterpret_cast<const int8_t *>(w) +
                                                                  (size_t)src * a.K + (size_t)c8 * 8));
            const float sc = __ldg(reinterpret_cast<const float *>(s) + src);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t word = i < 4 ? b.x : b.y;
                v[i] = (float)(int8_t)((word >> (8 * (i & 3))) & 0xFFu) * sc;
            }
        }
        uint4 o;
        o.x = h2_as_u32(__floats2half2_rn(v[0], v[1]));
        o.y = h2_as_u32(__floats2half2_rn(v[2], v[3]));
        o.z = h2_as_u32(__floats2half2_rn(v[4], v[5]));
        o.w = h2_as_u32(__floats2half2_rn(v[6], v[7]));
        *reinterpret_cast<uint4 *>(a.out + (size_t)r * a.K + (size_t)c8 * 8) = o;
    }
}

// ---------------------------------------------------------------------------
// Row kernels: one CTA per row.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_embed(const uint16_t *embed, const int *tokens, int h, float *x) {
    const int i = blockIdx.x;
    const uint16_t *src = embed + (size_t)__ldg(tokens + i) * h;
    for (int k = threadIdx.x; k < h; k += blockDim.x) x[(size_t)i * h + k] = bf16_bits_to_float(__ldg(src + k));
}

// One CTA per row: float4 loads kept in registers (rows up to 4096 wide),
// one block reduction, 8-byte stores of four fp16 outputs.
constexpr int kNormThreads = 128, kNormVec = 8;
__global__ void __launch_bounds__(kNormThreads) k_rmsnorm(const float *x, const uint16_t *gamma, float eps, int h,
                                                          uint16_t *out) {
    __shared__ float red[kNormThreads / 32];
    pdl_launch();  // the GEMM after this kernel may start its weight loads
    const float4 *row = reinterpret_cast<const float4 *>(x + (size_t)blockIdx.x * h);
    const int n4 = h >> 2;
    float4 v[kNormVec];
    float ss = 0.f;
    auto sq = [](const float4 &t) { return t.x * t.x + t.y * t.y + t.z * t.z + t.w * t.w; };
#pragma unroll
    for (int j = 0; j < kNormVec; ++j) {
        const int i = (int)threadIdx.x + j * kNormThreads;
        v[j] = i < n4 ? row[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        ss += sq(v[j]);
    }
    for (int i = (int)threadIdx.x + kNormVec * kNormThreads; i < n4; i += kNormThreads) ss += sq(row[i]);
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) t += red[w];
    const float inv = rsqrtf(t / (float)h + eps);
    const uint2 *g = reinterpret_cast<const uint2 *>(gamma);
    uint2 *o = reinterpret_cast<uint2 *>(out + (size_t)blockIdx.x * h);
    auto put = [&](int i, const float4 &a) {
        const uint2 gw = __ldg(g + i);
        const __half2 lo = __floats2half2_rn(bf16_bits_to_float((uint16_t)(gw.x & 0xFFFFu)) * (a.x * inv),
                                             bf16_bits_to_float((uint16_t)(gw.x >> 16)) * (a.y * inv));
        const __half2 hi = __floats2half2_rn(bf16_bits_to_float((uint16_t)(gw.y & 0xFFFFu)) * (a.z * inv),
                                             bf16_bits_to_float((uint16_t)(gw.y >> 16)) * (a.w * inv));
        o[i] = make_uint2(h2_as_u32(lo), h2_as_u32(hi));
    };
#pragma unroll
    for (int j = 0; j < kNormVec; ++j) {
        const int i = (int)threadIdx.x + j * kNormThreads;
        if (i < n4) put(i, v[j]);
    }
    for (int i = (int)threadIdx.x + kNormVec * kNormThreads; i < n4; i += kNormThreads) put(i, row[i]);
}

// One warp per (row, head): heads [0, Hq) queries, then Hkv keys, Hkv values.
template <int D>
__global__ void __launch_bounds__(128) k_qkv_rows(QkvRowsArgs a) {
    constexpr int M = D / 32;
    const int i = blockIdx.x;
    const int head = blockIdx.y * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    const int nh = a.Hq + 2 * a.Hkv;
    if (head >= nh) return;
    const int pos = a.pos0 + i;
    const bool is_q = head < a.Hq, is_k = !is_q && head < a.Hq + a.Hkv;
    const float *raw = a.raw + (size_t)i * nh * D + (size_t)head * D;
    const uint16_t *bias = is_q ? a.bq : (is_k ? a.bk : a.bv);
    const int hb = is_q ? head : (is_k ? head - a.Hq : head - a.Hq - a.Hkv);
    float v[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        v[m] = raw[lane + 32 * m];
        if (bias) v[m] += bf16_bits_to_float(__ldg(bias + (size_t)hb * D + lane + 32 * m));
    }
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
        // rotate_half pairs (j, j + D/2)
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
        uint16_t *qh = a.q_hi + ((size_t)i * a.Hq + head) * D, *ql = a.q_lo + ((size_t)i * a.Hq + head) * D;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const uint16_t hi = float_to_bf16_bits(v[m]);
            qh[lane + 32 * m] = hi;
            ql[lane + 32 * m] = float_to_bf16_bits(v[m] - bf16_bits_to_float(hi));
        }
        return;
    }
    const int phys = __ldg(a.page_table + pos / kPageTokens);
    if (phys < 0 || phys >= a.n_pages) {
        if (lane == 0 && a.err) atomicCAS(a.err, kErrNone, kErrBadPage);
        return;
    }
    uint16_t *dst = (is_k ? a.k_pool : a.v_pool) + (((size_t)phys * a.Hkv + hb) * kPageTokens + pos % kPageTokens) * D;
#pragma unroll
    for (int m = 0; m < M; ++m) dst[lane + 32 * m] = float_to_bf16_bits(v[m]);
}

// ---------------------------------------------------------------------------
// Causal flash attention.  CTA = (block of 64 query rows, query head h); warp
// w owns rows 16w .. 16w + 15.  Key blocks of 64 (4 pages) of KV head
// g = h / (Hq/Hkv) stream through a double-buffered cp.async ring with the
// 16-byte chunks of each row XOR-swizzled by (row & 7), so ldmatrix reads are
// conflict-free.  S = Q K^T and O += P V are mma.sync m16n8k16 contractions
// (bf16 in, fp32 accumulate) with Q and P as bf16 hi + lo pairs, so products
// carry ~16 significant bits; softmax is online in base 2.
// ---------------------------------------------------------------------------
QD_DEV uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
QD_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
QD_DEV void ldsm4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
QD_DEV void ldsm4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
QD_DEV void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
QD_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
QD_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
QD_DEV uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}
QD_DEV void split_bf16(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const float2 f = __bfloat1622float2(h);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = pack_bf16(a - f.x, b - f.y);
}

constexpr int kAttnRows = 64;   // query rows per CTA
constexpr int kAttnKeys = 64;   // keys per block

template <int D>
__global__ void __launch_bounds__(128) k_attn_rows(AttnRowsArgs a) {
    constexpr int CH = D / 8;            // 16-byte chunks per row
    constexpr int KS = D / 16;           // k-steps over d
    constexpr int NT = D / 8;            // n-tiles over d (output)
    extern __shared__ uint4 smem[];
    uint16_t *kv = reinterpret_cast<uint16_t *>(smem);  // [2 buffers][K, V][64 keys][D]
    pdl_launch();  // the o_proj GEMM after this kernel may start its weight loads
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
    const int h = blockIdx.y, g = h / (a.Hq / a.Hkv);
    const int q0 = blockIdx.x * kAttnRows;
    const int r_lo = q0 + 16 * warp + gq, r_hi = r_lo + 8;  // this thread's two query rows
    const int p_lo = a.pos0 + r_lo, p_hi = a.pos0 + r_hi;   // their positions
    const int T = a.pos0 + a.n;                              // keys that exist
    const int last = min(a.pos0 + q0 + kAttnRows - 1, T - 1);  // last key any row of the CTA needs
    const int n_blocks = last / kAttnKeys + 1;

    // query fragments (rows past n read row n - 1: computed, never written)
    uint32_t qh[KS][4], ql[KS][4];
    {
        const int ra = min(r_lo, a.n - 1), rb = min(r_hi, a.n - 1);
        const uint32_t *ha = reinterpret_cast<const uint32_t *>(a.q_hi + ((size_t)ra * a.Hq + h) * D);
        const uint32_t *hb = reinterpret_cast<const uint32_t *>(a.q_hi + ((size_t)rb * a.Hq + h) * D);
        const uint32_t *la = reinterpret_cast<const uint32_t *>(a.q_lo + ((size_t)ra * a.Hq + h) * D);
        const uint32_t *lb = reinterpret_cast<const uint32_t *>(a.q_lo + ((size_t)rb * a.Hq + h) * D);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            const int c = kk * 8 + tq;  // 32-bit word of dims 16kk + 2tq
            qh[kk][0] = __ldg(ha + c);
            qh[kk][1] = __ldg(hb + c);
            qh[kk][2] = __ldg(ha + c + 4);
            qh[kk][3] = __ldg(hb + c + 4);
            ql[kk][0] = __ldg(la + c);
            ql[kk][1] = __ldg(lb + c);
            ql[kk][2] = __ldg(la + c + 4);
            ql[kk][3] = __ldg(lb + c + 4);
        }
    }

    // K/V block b -> buffer b & 1 (keys past T or on a bad page read as zero)
    auto load_block = [&](int b) {
        uint16_t *ks = kv + (size_t)(b & 1) * 2 * kAttnKeys * D, *vs = ks + kAttnKeys * D;
        for (int u = threadIdx.x; u < kAttnKeys * CH; u += 128) {
            const int key = u / CH, ch = u % CH;
            const int kp = b * kAttnKeys + key;
            const uint32_t off = (uint32_t)(key * D + ((ch ^ (key & 7)) << 3)) * 2;
            int phys = -1;
            if (kp < T) {
                phys = __ldg(a.page_table + kp / kPageTokens);
                if (phys < 0 || phys >= a.n_pages) {
                    if (a.err) atomicCAS(a.err, kErrNone, kErrBadPage);
                    phys = -1;
                }
            }
            if (phys >= 0) {
                const size_t src = (((size_t)phys * a.Hkv + g) * kPageTokens + kp % kPageTokens) * D + ch * 8;
                cp_async16(smem_addr(ks) + off, a.k_pool + src);
                cp_async16(smem_addr(vs) + off, a.v_pool + src);
            } else {
                *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(ks) + off) = make_uint4(0, 0, 0, 0);
                *reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(vs) + off) = make_uint4(0, 0, 0, 0);
            }
        }
        cp_async_commit();
    };

    const float sscale = rsqrtf((float)D) * kLog2e;
    float o[NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;

    load_block(0);
    for (int b = 0; b < n_blocks; ++b) {
        if (b + 1 < n_blocks) {
            load_block(b + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint16_t *ks = kv + (size_t)(b & 1) * 2 * kAttnKeys * D, *vs = ks + kAttnKeys * D;
        const uint32_t ksa = smem_addr(ks), vsa = smem_addr(vs);

        // ---- S = Q K^T: 16 rows x 64 keys per warp
        float s[8][4];
#pragma unroll
        for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int key = 8 * j + (lane & 7);
#pragma unroll
            for (int kk = 0; kk < KS; kk += 2) {
                const int ch = 2 * kk + (lane >> 3);
                uint32_t b0, b1, b2, b3;
                ldsm4(ksa + (uint32_t)(key * D + ((ch ^ (key & 7)) << 3)) * 2, b0, b1, b2, b3);
                mma_bf16_16816(s[j], qh[kk][0], qh[kk][1], qh[kk][2], qh[kk][3], b0, b1);
                mma_bf16_16816(s[j], ql[kk][0], ql[kk][1], ql[kk][2], ql[kk][3], b0, b1);
                mma_bf16_16816(s[j], qh[kk + 1][0], qh[kk + 1][1], qh[kk + 1][2], qh[kk + 1][3], b2, b3);
                mma_bf16_16816(s[j], ql[kk + 1][0], ql[kk + 1][1], ql[kk + 1][2], ql[kk + 1][3], b2, b3);
            }
        }
        // ---- causal mask, online softmax (base 2)
        float mx_lo = m_lo, mx_hi = m_hi;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int kp = b * kAttnKeys + 8 * j + 2 * tq;
            s[j][0] = kp <= p_lo ? s[j][0] * sscale : -INFINITY;
            s[j][1] = kp + 1 <= p_lo ? s[j][1] * sscale : -INFINITY;
            s[j][2] = kp <= p_hi ? s[j][2] * sscale : -INFINITY;
            s[j][3] = kp + 1 <= p_hi ? s[j][3] * sscale : -INFINITY;
            mx_lo = fmaxf(mx_lo, fmaxf(s[j][0], s[j][1]));
            mx_hi = fmaxf(mx_hi, fmaxf(s[j][2], s[j][3]));
        }
#pragma unroll
        for (int o2 = 1; o2 < 4; o2 <<= 1) {
            mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, o2));
            mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, o2));
        }
        // rows with no visible key yet keep m = -inf: use 0 as the reference
        const float ref_lo = mx_lo == -INFINITY ? 0.f : mx_lo, ref_hi = mx_hi == -INFINITY ? 0.f : mx_hi;
        const float c_lo = exp2f(m_lo - ref_lo), c_hi = exp2f(m_hi - ref_hi);
        m_lo = mx_lo;
        m_hi = mx_hi;
        float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            s[j][0] = exp2f(s[j][0] - ref_lo);
            s[j][1] = exp2f(s[j][1] - ref_lo);
            s[j][2] = exp2f(s[j][2] - ref_hi);
            s[j][3] = exp2f(s[j][3] - ref_hi);
            sum_lo += s[j][0] + s[j][1];
            sum_hi += s[j][2] + s[j][3];
        }
        l_lo = l_lo * c_lo + sum_lo;
        l_hi = l_hi * c_hi + sum_hi;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            o[j][0] *= c_lo;
            o[j][1] *= c_lo;
            o[j][2] *= c_hi;
            o[j][3] *= c_hi;
        }
        // ---- O += P V: P as A fragments (k = keys), V via transposed ldmatrix
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t ph[4], pl[4];
            split_bf16(s[2 * kk][0], s[2 * kk][1], ph[0], pl[0]);
            split_bf16(s[2 * kk][2], s[2 * kk][3], ph[1], pl[1]);
            split_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1], ph[2], pl[2]);
            split_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3], ph[3], pl[3]);
            const int key = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int j = 0; j < NT; j += 2) {
                const int ch = j + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm4_t(vsa + (uint32_t)(key * D + ((ch ^ (key & 7)) << 3)) * 2, b0, b1, b2, b3);
                mma_bf16_16816(o[j], ph[0], ph[1], ph[2], ph[3], b0, b1);
                mma_bf16_16816(o[j], pl[0], pl[1], pl[2], pl[3], b0, b1);
                mma_bf16_16816(o[j + 1], ph[0], ph[1], ph[2], ph[3], b2, b3);
                mma_bf16_16816(o[j + 1], pl[0], pl[1], pl[2], pl[3], b2, b3);
            }
        }
        __syncthreads();  // the buffer is refilled two blocks later
    }
#pragma unroll
    for (int o2 = 1; o2 < 4; o2 <<= 1) {
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, o2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, o2);
    }
    const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f, inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
    const size_t ld = (size_t)a.Hq * D;
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int col = h * D + 8 * j + 2 * tq;
        if (r_lo < a.n)
            *reinterpret_cast<half2 *>(a.out + (size_t)r_lo * ld + col) =
                __floats2half2_rn(o[j][0] * inv_lo, o[j][1] * inv_lo);
        if (r_hi < a.n)
            *reinterpret_cast<half2 *>(a.out + (size_t)r_hi * ld + col) =
                __floats2half2_rn(o[j][2] * inv_hi, o[j][3] * inv_hi);
    }
}

}  // namespace

cudaError_t launch_dequant(cudaStream_t stream, int n_sm, const DequantArgs &a) {
    if (!a.w || !a.s || !a.out || a.N <= 0 || a.K <= 0 || a.K % 8) return cudaErrorInvalidValue;
    if (a.fmt == kFmtInt4 ? a.K % kGroup != 0 : a.fmt != kFmtInt8) return cudaErrorInvalidValue;
    if (a.w2 && (!a.s2 || a.N % 64)) return cudaErrorInvalidValue;
    const long long units = (long long)(a.w2 ? 2 : 1) * a.N * (a.K / 8);
    const long long want = (units + 255) / 256;
    const int grid = (int)(want < 8LL * n_sm ? want : 8LL * n_sm);
    k_dequant<<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_embed_rows(cudaStream_t stream, const uint16_t *embed, const int *tokens, int n, int h,
                              float *x) {
    if (n <= 0) return cudaErrorInvalidValue;
    k_embed<<<n, 256, 0, stream>>>(embed, tokens, h, x);
    return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rows(cudaStream_t stream, const float *x, const uint16_t *gamma, float eps, int n,
                                int h, uint16_t *out) {
    if (n <= 0 || h <= 0 || h % 4 || ((uintptr_t)x & 15) || ((uintptr_t)gamma & 7) || ((uintptr_t)out & 7))
        return cudaErrorInvalidValue;
    k_rmsnorm<<<n, kNormThreads, 0, stream>>>(x, gamma, eps, h, out);
    return cudaGetLastError();
}

cudaError_t launch_qkv_rows(cudaStream_t stream, const QkvRowsArgs &a) {
    if (a.n <= 0 || (a.d != 64 && a.d != 128)) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)a.n, (unsigned)((a.Hq + 2 * a.Hkv + 3) / 4));
    if (a.d == 128)
        k_qkv_rows<128><<<grid, 128, 0, stream>>>(a);
    else
        k_qkv_rows<64><<<grid, 128, 0, stream>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_attn_rows(cudaStream_t stream, const AttnRowsArgs &a) {
    if (a.n <= 0 || (a.d != 64 && a.d != 128) || a.Hq % a.Hkv) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((a.n + kAttnRows - 1) / kAttnRows), (unsigned)a.Hq);
    const size_t smem = (size_t)2 * 2 * kAttnKeys * a.d * 2;
    LaunchCfg lc{};
    lc.stream = stream;
    if (a.d == 128) return launch_k(lc, k_attn_rows<128>, grid, dim3(128), smem, a);
    return launch_k(lc, k_attn_rows<64>, grid, dim3(128), smem, a);
}

}  // namespace qd
