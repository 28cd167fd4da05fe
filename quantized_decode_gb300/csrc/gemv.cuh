// gemv.cuh - weight-streaming dequant dot products for the batch-1 decode GEMVs.
//
// Work unit: 16 bytes of one weight row (32 INT4 codes, 16 INT8 codes or 8
// bf16 values), loaded with one 128-bit streaming load.  A warp is split into
// 32/LPR row slots of LPR lanes; the lanes of a slot stride over the units of
// their rows and every lane carries RT rows at once, so one shared-memory load
// of the activations serves RT weight rows.  The LPR partial sums of a row are
// then combined with shuffles.
//
// Activations are staged in shared memory as fp16 pairs scaled by a power of
// two 2^-e chosen so that every |value| <= 1 (fp16 products and short fp16 sums
// then cannot overflow); the result is multiplied back by 2^e in fp32.
#pragma once

#include "common.cuh"

namespace qd {

// ---------------------------------------------------------------------------
// INT4 ValueShuffle word -> four exact fp16 code pairs.
// The word holds codes c0..c7 at bit shifts 0,16,4,20,8,24,12,28, so the
// half-words carry the pairs (c0,c1) at bits (0,16), (c2,c3) at (4,20),
// (c4,c5) at (8,24) and (c6,c7) at (12,28).  For a two's-complement nibble,
// nibble ^ 8 = c + 8 in [0, 15]:
//   ((w & 0x000F000F) ^ 0x64086408) is the fp16 pair 1024 + (c + 8)      -> minus 1032
//   ((w & 0x00F000F0) ^ 0x64806480) is the fp16 pair 1024 + 16 (c + 8)   -> /16 - 72
// Both corrections are exact, so the pairs equal the codes exactly.
// ---------------------------------------------------------------------------
QD_DEV half2 int4_word_dot(uint32_t w, uint4 xq, half2 acc) {
    const half2 k1032 = u32_as_h2(0x64086408u);   // (1032, 1032)
    const half2 kSixteenth = u32_as_h2(0x2C002C00u);  // (1/16, 1/16)
    const half2 kNeg72 = u32_as_h2(0xD480D480u);  // (-72, -72)
    const uint32_t w8 = w >> 8;
    const half2 c01 = __hsub2(u32_as_h2(lop3_and_xor(w, 0x000F000Fu, 0x64086408u)), k1032);
    const half2 c23 = __hfma2(u32_as_h2(lop3_and_xor(w, 0x00F000F0u, 0x64806480u)), kSixteenth, kNeg72);
    const half2 c45 = __hsub2(u32_as_h2(lop3_and_xor(w8, 0x000F000Fu, 0x64086408u)), k1032);
    const half2 c67 = __hfma2(u32_as_h2(lop3_and_xor(w8, 0x00F000F0u, 0x64806480u)), kSixteenth, kNeg72);
    acc = __hfma2(c01, u32_as_h2(xq.x), acc);
    acc = __hfma2(c23, u32_as_h2(xq.y), acc);
    acc = __hfma2(c45, u32_as_h2(xq.z), acc);
    acc = __hfma2(c67, u32_as_h2(xq.w), acc);
    return acc;
}

// INT8 word (codes b0..b3 in natural byte order) -> two exact fp16 pairs.
// b ^ 0x80 = c + 128 in [1, 255]; placing it under the fp16 exponent of 1024
// with a byte permute gives 1024 + c + 128, and subtracting 1152 is exact.
QD_DEV half2 int8_word_dot(uint32_t w, uint32_t x01, uint32_t x23, half2 acc) {
    const half2 k1152 = u32_as_h2(0x64806480u);
    const uint32_t t = w ^ 0x80808080u;
    const half2 c01 = __hsub2(u32_as_h2(prmt(t, 0x64646464u, 0x4140u)), k1152);
    const half2 c23 = __hsub2(u32_as_h2(prmt(t, 0x64646464u, 0x4342u)), k1152);
    acc = __hfma2(c01, u32_as_h2(x01), acc);
    acc = __hfma2(c23, u32_as_h2(x23), acc);
    return acc;
}

QD_DEV float h2_sum(half2 a, half2 b) {
    const float2 fa = __half22float2(a), fb = __half22float2(b);
    return (fa.x + fa.y) + (fb.x + fb.y);
}

// Packed fp32 FMA on two lanes (Blackwell fma.rn.f32x2).
QD_DEV float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// ---------------------------------------------------------------------------
// Row-tile dot products.  wrow[i]: the 16-byte units of row i; xs4: staged
// activations; U: units per row; j: this lane's index within its slot.
// On return every lane of the slot holds the full dot product of each row
// (in the prescaled units of the staged activations).
// ---------------------------------------------------------------------------

// INT4 group-128: unit u covers codes 32u..32u+31, group u/4; scale per (row, group).
template <int LPR, int RT>
QD_DEV void int4_tile_dots(const uint4 *const (&wrow)[RT], const uint16_t *const (&srow)[RT],
                           const uint4 *__restrict__ xs4, int U, int j, float (&out)[RT]) {
    float acc[RT];
#pragma unroll
    for (int i = 0; i < RT; ++i) acc[i] = 0.f;
    uint4 cur[RT];
    uint16_t scur[RT];
    int u = j;
    if (u < U) {
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            cur[i] = ld_stream(wrow[i] + u);
            scur[i] = __ldg(srow[i] + (u >> 2));
        }
    }
    for (; u < U; u += LPR) {
        uint4 nxt[RT];
        uint16_t snxt[RT];
        const int un = u + LPR;
        if (un < U) {
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                nxt[i] = ld_stream(wrow[i] + un);
                snxt[i] = __ldg(srow[i] + (un >> 2));
            }
        }
        const uint4 x0 = xs4[4 * u + 0], x1 = xs4[4 * u + 1];
        const uint4 x2 = xs4[4 * u + 2], x3 = xs4[4 * u + 3];
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            half2 a = u32_as_h2(0u), b = u32_as_h2(0u);
            a = int4_word_dot(cur[i].x, x0, a);
            b = int4_word_dot(cur[i].y, x1, b);
            a = int4_word_dot(cur[i].z, x2, a);
            b = int4_word_dot(cur[i].w, x3, b);
            acc[i] = fmaf(h2_sum(a, b), bf16_bits_to_float(scur[i]), acc[i]);
        }
        if (un < U) {
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                cur[i] = nxt[i];
                scur[i] = snxt[i];
            }
        }
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) out[i] = slot_sum<LPR>(acc[i]);
}

// INT8 per-row: unit u covers codes 16u..16u+15; the row scale is applied by the caller.
template <int LPR, int RT>
QD_DEV void int8_tile_dots(const uint4 *const (&wrow)[RT], const uint4 *__restrict__ xs4, int U,
                           int j, float (&out)[RT]) {
    float acc[RT];
#pragma unroll
    for (int i = 0; i < RT; ++i) acc[i] = 0.f;
    uint4 cur[RT];
    int u = j;
    if (u < U) {
#pragma unroll
        for (int i = 0; i < RT; ++i) cur[i] = ld_stream(wrow[i] + u);
    }
    for (; u < U; u += LPR) {
        uint4 nxt[RT];
        const int un = u + LPR;
        if (un < U) {
#pragma unroll
            for (int i = 0; i < RT; ++i) nxt[i] = ld_stream(wrow[i] + un);
        }
        const uint4 x0 = xs4[2 * u + 0], x1 = xs4[2 * u + 1];
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            half2 a = u32_as_h2(0u), b = u32_as_h2(0u);
            a = int8_word_dot(cur[i].x, x0.x, x0.y, a);
            b = int8_word_dot(cur[i].y, x0.z, x0.w, b);
            a = int8_word_dot(cur[i].z, x1.x, x1.y, a);
            b = int8_word_dot(cur[i].w, x1.z, x1.w, b);
            acc[i] += h2_sum(a, b);
        }
        if (un < U) {
#pragma unroll
            for (int i = 0; i < RT; ++i) cur[i] = nxt[i];
        }
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) out[i] = slot_sum<LPR>(acc[i]);
}

// bf16 rows against fp32 activations (LM head): unit u covers values 8u..8u+7.
template <int LPR, int RT>
QD_DEV void bf16_tile_dots(const uint4 *const (&wrow)[RT], const float4 *__restrict__ xs,
                           int U, int j, float (&out)[RT]) {
    float2 acc[RT];
#pragma unroll
    for (int i = 0; i < RT; ++i) acc[i] = make_float2(0.f, 0.f);
    uint4 cur[RT];
    int u = j;
    if (u < U) {
#pragma unroll
        for (int i = 0; i < RT; ++i) cur[i] = ld_stream(wrow[i] + u);
    }
    for (; u < U; u += LPR) {
        uint4 nxt[RT];
        const int un = u + LPR;
        if (un < U) {
#pragma unroll
            for (int i = 0; i < RT; ++i) nxt[i] = ld_stream(wrow[i] + un);
        }
        const float4 xa = xs[2 * u], xb = xs[2 * u + 1];
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            const uint4 w = cur[i];
            acc[i] = ffma2(make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u)),
                           make_float2(xa.x, xa.y), acc[i]);
            acc[i] = ffma2(make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u)),
                           make_float2(xa.z, xa.w), acc[i]);
            acc[i] = ffma2(make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xFFFF0000u)),
                           make_float2(xb.x, xb.y), acc[i]);
            acc[i] = ffma2(make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xFFFF0000u)),
                           make_float2(xb.z, xb.w), acc[i]);
        }
        if (un < U) {
#pragma unroll
            for (int i = 0; i < RT; ++i) cur[i] = nxt[i];
        }
    }
#pragma unroll
    for (int i = 0; i < RT; ++i) out[i] = slot_sum<LPR>(acc[i].x + acc[i].y);
}

// ---------------------------------------------------------------------------
// Activation staging (block-wide; every thread calls).
// src: fp32 [K] (src_bf16 == nullptr) or bf16 [K]; gamma: bf16 RMSNorm gain or
// nullptr (no norm).  K % 4 == 0.
//   half_out: fp16 pairs of gamma*x*inv_rms*2^-e, max |value| < 1; returns 2^e.
//   f32_out:  fp32 gamma*x*inv_rms (no prescale); returns 1.
// red: shared scratch of 2*32 floats.
// ---------------------------------------------------------------------------
template <int NT>
QD_DEV float stage_activations(const float *__restrict__ src, const uint16_t *__restrict__ src_bf16,
                               const uint16_t *__restrict__ gamma, float eps, int K,
                               half2 *half_out, float *f32_out, float *red) {
    const int tid = threadIdx.x;
    auto load4 = [&](int i) -> float4 {
        if (src_bf16) {
            const uint2 b = *reinterpret_cast<const uint2 *>(src_bf16 + i);
            return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                               __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
        }
        return __ldcg(reinterpret_cast<const float4 *>(src + i));
    };
    auto gain4 = [&](int i) -> float4 {
        if (!gamma) return make_float4(1.f, 1.f, 1.f, 1.f);
        const uint2 b = __ldg(reinterpret_cast<const uint2 *>(gamma + i));
        return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                           __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
    };
    float ss = 0.f, mx = 0.f;
    for (int i = tid * 4; i < K; i += NT * 4) {
        const float4 v = load4(i), g = gain4(i);
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x * g.x), fabsf(v.y * g.y)),
                             fmaxf(fabsf(v.z * g.z), fabsf(v.w * g.w))));
    }
    ss = warp_sum(ss);
    mx = warp_max(mx);
    const int warp = tid >> 5, lane = tid & 31;
    if (lane == 0) {
        red[warp] = ss;
        red[32 + warp] = mx;
    }
    __syncthreads();
    if (warp == 0) {
        float a = lane < NT / 32 ? red[lane] : 0.f;
        float b = lane < NT / 32 ? red[32 + lane] : 0.f;
        a = warp_sum(a);
        b = warp_max(b);
        if (lane == 0) {
            red[0] = a;
            red[32] = b;
        }
    }
    __syncthreads();
    const float inv = gamma ? rsqrtf(red[0] / (float)K + eps) : 1.f;
    float post = 1.f, pre = inv;
    if (half_out) {
        const float amax = red[32] * inv;
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        pre = ldexpf(inv, -e);
        post = ldexpf(1.f, e);
    }
    for (int i = tid * 4; i < K; i += NT * 4) {
        const float4 v = load4(i), g = gain4(i);
        if (half_out) {
            half_out[i / 2] = __floats2half2_rn(g.x * (v.x * pre), g.y * (v.y * pre));
            half_out[i / 2 + 1] = __floats2half2_rn(g.z * (v.z * pre), g.w * (v.w * pre));
        } else {
            *reinterpret_cast<float4 *>(f32_out + i) =
                make_float4(g.x * (v.x * pre), g.y * (v.y * pre), g.z * (v.z * pre), g.w * (v.w * pre));
        }
    }
    __syncthreads();
    return post;
}

}  // namespace qd
