// gemv.cuh - weight-streaming dequant dot products for the batch-1 decode GEMVs.
//
// Work unit: 16 bytes of one weight row (32 INT4 codes, 16 INT8 codes or 8
// bf16 values).  A warp is split into 32/LPR row slots of LPR lanes; the lanes
// of a slot stride over the units of their rows and every lane carries RT rows
// at once, so one shared-memory load of the activations serves RT weight rows.
// The LPR partial sums of a row are then combined with shuffles.
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

// Swizzle of staged activations (see stage_activations): the staged vector is
// cut into blocks of one weight unit's activations (blk_bytes = 64 for INT4
// units of 32 codes as fp16, 32 for INT8 units as fp16 and for bf16 units as
// fp32) and the 16-byte chunks of a block are XOR-permuted by block-index bits,
// so the 8 lanes of a row slot, which read the same chunk of 8 consecutive
// blocks, hit distinct bank groups.
QD_HOST_DEV_INLINE uint32_t swz_mask(uint32_t blk, int blk_bytes) {
    return blk_bytes == 64 ? ((blk >> 1) & 3u) : ((blk >> 2) & 1u);
}
QD_DEV uint32_t swz_offset(uint32_t byte_off, int blk_bytes) {
    if (blk_bytes == 0) return byte_off;
    const uint32_t blk = byte_off / (uint32_t)blk_bytes, in = byte_off % (uint32_t)blk_bytes;
    return blk * (uint32_t)blk_bytes + ((((in >> 4) ^ swz_mask(blk, blk_bytes))) << 4) + (in & 15u);
}
template <int FMT>
constexpr int act_blk_bytes() {
    return FMT == kFmtInt4 ? 64 : 32;
}

// ---------------------------------------------------------------------------
// Weight streaming through a lane-private shared-memory ring.
//
// A warp owns row tiles t_first, t_first + t_stride, ... < n_tiles and, within
// each of them, the slabs [sb_begin, sb_end) of its K part; a slab is 16
// consecutive 16-byte units of a row (512 INT4 codes, 256 INT8 codes or 128
// bf16 values).  A row slot is 8 lanes; lane j takes units 16 s + j and
// 16 s + 8 + j of slab s, so each copy instruction covers 128 contiguous bytes
// of every row.  Every lane carries RT rows (rows(tile, i): their units and,
// for INT4, their scale rows), so one shared-memory read of the activations
// serves RT rows.  Units past the end of a row (K not a multiple of a slab)
// are skipped.
//
// Each lane copies exactly the bytes it will consume (cp.async: two 16-byte
// units per row and step) into its own slots of a D-stage ring, D - 1 steps
// ahead of the arithmetic, one commit group per step; the ring flows across
// tile boundaries, and since a lane only reads what its row slot copied, no
// barrier is needed beyond the warp's own.  For INT4 the 16 units of a row's
// slab share 4 bf16 group scales (8 bytes, two aligned words: the row's scales
// start 4-byte aligned as groups per row are even), which lanes 0 and 1 of the
// row slot copy once per step.
// At the end of a tile the 8 partial sums of each row are combined with
// shuffles and `epi(tile, out)` runs on every lane (all lanes of a row slot
// hold the same sums).  `sync()` (the dependency wait and the activation
// staging) runs on all threads once, after the ring's first D - 1 steps of
// weight copies are on their way.
//
// Ring layout per warp: stage s, row i, unit h, lane l -> 16-byte unit at
// ring[((s * RT + i) * 2 + h) * 32 + l]; row slot r's scale word w (groups
// 4 slab + 2w, +1) at sring[((s * RT + i) * 4 + r) * 2 + w].
// ---------------------------------------------------------------------------
constexpr int kLanesPerRow = 8;

struct RowRef {
    const uint4 *w;     // 16-byte units of the row
    const uint16_t *s;  // INT4: bf16 scales of the row, one per 128 codes
};


template <int RT, int D>
constexpr size_t code_ring_bytes_per_warp() {
    return (size_t)D * RT * 2 * 32 * 16;
}
template <int RT, int D>
constexpr size_t scale_ring_words_per_warp() {
    return (size_t)D * RT * 8;
}
template <int RT, int D>
constexpr size_t ring_bytes_per_warp() {
    return code_ring_bytes_per_warp<RT, D>() + scale_ring_words_per_warp<RT, D>() * 4;
}
// Warp `warp`'s code and scale rings in a block of NW warps' rings at `base`
// (all code rings first, 16-byte aligned, then all scale rings).
template <int RT, int D>
QD_DEV void warp_rings(void *base, int NW, int warp, uint4 *&ring, uint32_t *&sring) {
    ring = reinterpret_cast<uint4 *>(base) + (size_t)warp * (code_ring_bytes_per_warp<RT, D>() / 16);
    sring = reinterpret_cast<uint32_t *>(reinterpret_cast<char *>(base) + (size_t)NW * code_ring_bytes_per_warp<RT, D>()) +
            (size_t)warp * scale_ring_words_per_warp<RT, D>();
}

// One 16-byte unit of a row against its staged activations (x: 4 chunks for
// INT4 as fp16, 2 chunks for INT8 as fp16, 2 float4 for bf16), fp32 result.
QD_DEV float int4_unit_dot(uint4 q, const uint4 (&x)[4]) {
    half2 a = u32_as_h2(0u), b = u32_as_h2(0u);
    a = int4_word_dot(q.x, x[0], a);
    b = int4_word_dot(q.y, x[1], b);
    a = int4_word_dot(q.z, x[2], a);
    b = int4_word_dot(q.w, x[3], b);
    const float2 f = __half22float2(__hadd2(a, b));
    return f.x + f.y;
}
// INT4 unit against int8 activations (kFmtInt4A8): the word's nibbles n = c + 8
// as bytes -- (w & 0x0F0F0F0F) ^ 0x08080808 holds n0, n4, n1, n5 and the same of
// w >> 4 holds n2, n6, n3, n7 -- against activation bytes staged in that order
// (q0 q4 q1 q5 | q2 q6 q3 q7 per 8 codes); returns sum n q (exact), the caller
// subtracts 8 sum q.
QD_DEV int int4_a8_unit_dot(uint4 q, const uint4 (&x)[2]) {
    int s = 0;
    s = __dp4a((int)lop3_and_xor(q.x, 0x0F0F0F0Fu, 0x08080808u), (int)x[0].x, s);
    s = __dp4a((int)lop3_and_xor(q.x >> 4, 0x0F0F0F0Fu, 0x08080808u), (int)x[0].y, s);
    s = __dp4a((int)lop3_and_xor(q.y, 0x0F0F0F0Fu, 0x08080808u), (int)x[0].z, s);
    s = __dp4a((int)lop3_and_xor(q.y >> 4, 0x0F0F0F0Fu, 0x08080808u), (int)x[0].w, s);
    s = __dp4a((int)lop3_and_xor(q.z, 0x0F0F0F0Fu, 0x08080808u), (int)x[1].x, s);
    s = __dp4a((int)lop3_and_xor(q.z >> 4, 0x0F0F0F0Fu, 0x08080808u), (int)x[1].y, s);
    s = __dp4a((int)lop3_and_xor(q.w, 0x0F0F0F0Fu, 0x08080808u), (int)x[1].z, s);
    s = __dp4a((int)lop3_and_xor(q.w >> 4, 0x0F0F0F0Fu, 0x08080808u), (int)x[1].w, s);
    return s;
}
QD_DEV float int8_unit_dot(uint4 q, const uint4 (&x)[2]) {
    half2 a = u32_as_h2(0u), b = u32_as_h2(0u);
    a = int8_word_dot(q.x, x[0].x, x[0].y, a);
    b = int8_word_dot(q.y, x[0].z, x[0].w, b);
    a = int8_word_dot(q.z, x[1].x, x[1].y, a);
    b = int8_word_dot(q.w, x[1].z, x[1].w, b);
    const float2 f = __half22float2(__hadd2(a, b));
    return f.x + f.y;
}
QD_DEV float bf16_unit_dot(uint4 q, const float4 (&x)[2]) {
    float2 p = make_float2(0.f, 0.f);
    p = ffma2(make_float2(__uint_as_float(q.x << 16), __uint_as_float(q.x & 0xFFFF0000u)), make_float2(x[0].x, x[0].y), p);
    p = ffma2(make_float2(__uint_as_float(q.y << 16), __uint_as_float(q.y & 0xFFFF0000u)), make_float2(x[0].z, x[0].w), p);
    p = ffma2(make_float2(__uint_as_float(q.z << 16), __uint_as_float(q.z & 0xFFFF0000u)), make_float2(x[1].x, x[1].y), p);
    p = ffma2(make_float2(__uint_as_float(q.w << 16), __uint_as_float(q.w & 0xFFFF0000u)), make_float2(x[1].z, x[1].w), p);
    return p.x + p.y;
}

template <int FMT, int RT, int D, class Rows, class Epi, class Sync>
QD_DEV void gemv_stream(const Rows &rows, const Epi &epi, const Sync &sync, int t_first, int t_stride,
                        int n_tiles, int sb_begin, int sb_end, int U, int j, const void *xs, uint4 *ring,
                        uint32_t *sring, const float *a8_sx = nullptr, const int *a8_qs = nullptr) {
    static_assert(D >= 2, "ring depth");
    constexpr bool W4 = FMT == kFmtInt4 || FMT == kFmtInt4A8;  // INT4 codes and group scales
    constexpr int XC = FMT == kFmtInt4 ? 4 : 2;  // 16-byte activation chunks per unit
    const int lane = threadIdx.x & 31;
    const int n_it = sb_end > sb_begin ? sb_end - sb_begin : 0;
    const int my_tiles = t_first < n_tiles ? (n_tiles - 1 - t_first) / t_stride + 1 : 0;
    const int F = my_tiles * n_it;

    const uint32_t xm = swz_mask((uint32_t)j, act_blk_bytes<FMT>());  // same for both units of every slab

    int lt = t_first, li = 0;  // load cursor
    RowRef lrow[RT];
    auto load_rows = [&](int t) {
#pragma unroll
        for (int i = 0; i < RT; ++i) lrow[i] = rows(t, i);
    };
    if (F > 0) load_rows(lt);
    const int rslot = lane / kLanesPerRow;
    auto issue = [&](int f) {
        const int slot = f % D;
        const int sb = sb_begin + li;
        const int ub = 16 * sb + j;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int u = ub + 8 * h;
            if (u < U) {
#pragma unroll
                for (int i = 0; i < RT; ++i) cp_async16(ring + ((slot * RT + i) * 2 + h) * 32 + lane, lrow[i].w + u);
            }
        }
        if constexpr (W4) {
            // lane j < 2 of the slot: word j of the slab's 4 group scales (groups per row: U / 4, even)
            if (j < 2 && 4 * sb + 2 * j < (U >> 2)) {
#pragma unroll
                for (int i = 0; i < RT; ++i)
                    cp_async4(sring + ((slot * RT + i) * 4 + rslot) * 2 + j, lrow[i].s + 4 * sb + 2 * j);
            }
        }
        if (++li == n_it) {
            li = 0;
            lt += t_stride;
            if (lt < n_tiles) load_rows(lt);
        }
    };
    // The first D - 1 steps of weights go out before the dependency wait:
    // nothing an earlier kernel writes is read by them, so under programmatic
    // dependent launch they overlap the previous kernel's tail.
    for (int s = 0; s < D - 1; ++s) {
        if (s < F) issue(s);
        cp_async_commit();
    }
    sync();

    float acc[RT];
#pragma unroll
    for (int i = 0; i < RT; ++i) acc[i] = 0.f;
    int ct = t_first, ci = 0;  // compute cursor
    const bool shi = (j >> 2) != 0;  // the unit's group scale is the high half of its word
#pragma unroll 1
    for (int f = 0; f < F; ++f) {
        // the scale words are shared by the lanes of a row slot: every lane is
        // past its reads of the stage before it is refilled (here), and sees the
        // copying lanes' words once they completed (after the wait)
        if constexpr (W4) __syncwarp();
        if (f + D - 1 < F) issue(f + D - 1);
        cp_async_commit();
        cp_async_wait<D - 1>();
        if constexpr (W4) __syncwarp();
        const int slot = f % D;
        const int ub = 16 * (sb_begin + ci) + j;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int u = ub + 8 * h;
            if (u < U) {
                if constexpr (FMT == kFmtBf16) {
                    const float4 *x4 = reinterpret_cast<const float4 *>(xs) + XC * u;
                    float4 xr[2];
#pragma unroll
                    for (int k = 0; k < 2; ++k) xr[k] = x4[k ^ xm];
#pragma unroll
                    for (int i = 0; i < RT; ++i) acc[i] += bf16_unit_dot(ring[((slot * RT + i) * 2 + h) * 32 + lane], xr);
                } else {
                    const uint4 *x4 = reinterpret_cast<const uint4 *>(xs) + XC * u;
                    uint4 xr[XC];
#pragma unroll
                    for (int k = 0; k < XC; ++k) xr[k] = x4[k ^ xm];
#pragma unroll
                    for (int i = 0; i < RT; ++i) {
                        const int idx = ((slot * RT + i) * 2 + h) * 32 + lane;
                        if constexpr (FMT == kFmtInt4) {
                            const uint32_t sw = sring[((slot * RT + i) * 4 + rslot) * 2 + h];
                            const float sc = __uint_as_float(shi ? (sw & 0xFFFF0000u) : (sw << 16));
                            acc[i] = fmaf(int4_unit_dot(ring[idx], xr), sc, acc[i]);
                        } else if constexpr (FMT == kFmtInt4A8) {
                            const uint32_t sw = sring[((slot * RT + i) * 4 + rslot) * 2 + h];
                            const float sc = __uint_as_float(shi ? (sw & 0xFFFF0000u) : (sw << 16));
                            const int d = int4_a8_unit_dot(ring[idx], xr) - 8 * a8_qs[u];
                            acc[i] = fmaf((float)d, sc * a8_sx[u >> 2], acc[i]);
                        } else {
                            acc[i] += int8_unit_dot(ring[idx], xr);
                        }
                    }
                }
            }
        }
        if (++ci == n_it) {
            float out[RT];
#pragma unroll
            for (int i = 0; i < RT; ++i) {
                out[i] = slot_sum<kLanesPerRow>(acc[i]);
                acc[i] = 0.f;
            }
            epi(ct, out);
            ci = 0;
            ct += t_stride;
        }
    }
    cp_async_wait<0>();
}

// Sum of K-part partials for a tile shared by KS warps of one CTA (named barrier
// per tile slot).  Every warp calls it with its partial; the warp of part 0
// returns true with the totals in out.  red: KS * 32 * RT floats for this slot.
template <int RT>
QD_DEV bool ksplit_reduce(float (&out)[RT], int ks, int kp, int slot_id, float *red, int j, int row_slot,
                          int lpr) {
    if (ks == 1) return true;
    const int lane = threadIdx.x & 31;
    if (j == 0) {
#pragma unroll
        for (int i = 0; i < RT; ++i) red[(kp * 32 + row_slot) * RT + i] = out[i];
    }
    asm volatile("bar.sync %0, %1;" ::"r"(1 + slot_id), "r"(ks * 32) : "memory");
    bool mine = kp == 0;
    if (mine) {
#pragma unroll
        for (int i = 0; i < RT; ++i) {
            float v = 0.f;
            for (int q = 0; q < ks; ++q) v += red[(q * 32 + row_slot) * RT + i];
            out[i] = v;
        }
    }
    asm volatile("bar.sync %0, %1;" ::"r"(1 + slot_id), "r"(ks * 32) : "memory");
    (void)lane;
    (void)lpr;
    return mine;
}

// Units per row for a weight format: 16 bytes hold 32 INT4, 16 INT8 or 8 bf16 values.
QD_HOST_DEV_INLINE bool int4_weights(int fmt) { return fmt == kFmtInt4 || fmt == kFmtInt4A8; }
QD_HOST_DEV_INLINE int units_per_row(int fmt, int K) {
    return int4_weights(fmt) ? K / 32 : (fmt == kFmtInt8 ? K / 16 : K / 8);
}

// Slabs (16 units) per row, the last one possibly partial.
QD_HOST_DEV_INLINE int slabs_per_row(int fmt, int K) { return (units_per_row(fmt, K) + 15) / 16; }

// ---------------------------------------------------------------------------
// Activation statistics handed from producer to consumer.
//
// A kernel that writes the vector the next kernel consumes also reduces, over
// the elements its CTA wrote, the sum of squares and max |value * gamma_next|
// (gamma_next: the consumer's RMSNorm gain, or none) into one (ss, mx) pair per
// CTA in a fixed array of kStatSlots pairs.  Slots of CTAs that a launch does
// not have stay zero, which is neutral for both the sum and the max.  The
// consumer then needs a single pass over its input.
// ---------------------------------------------------------------------------
// Block-wide reduction of per-thread (ss, mx) into out[2 * blockIdx.x + {0, 1}].
QD_DEV void write_block_stats(float ss, float mx, float *out, float *red) {
    ss = warp_sum(ss);
    mx = warp_max(mx);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = (blockDim.x + 31) >> 5;
    __syncthreads();
    if (lane == 0) {
        red[warp] = ss;
        red[32 + warp] = mx;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float a = 0.f, b = 0.f;
        for (int w = 0; w < nw; ++w) {
            a += red[w];
            b = fmaxf(b, red[32 + w]);
        }
        out[2 * blockIdx.x] = a;
        out[2 * blockIdx.x + 1] = b;
    }
}

// ---------------------------------------------------------------------------
// Activation staging (block-wide; every thread calls).
// src: fp32 [K] (src_bf16 == nullptr) or bf16 [K]; gamma: bf16 RMSNorm gain or
// nullptr (no norm).  K % 4 == 0.  With stats_in (kStatSlots producer pairs)
// the sum of squares and max |x*gamma| come from the producer and the input
// is read once; otherwise they are computed here first.
//   half_out: fp16 pairs of gamma*x*inv_rms*2^-e, max |value| < 1; returns 2^e.
//   f32_out:  fp32 gamma*x*inv_rms (no prescale); returns 1.
//   i8_out:   (kFmtInt4A8) the fp32 values gamma*x*inv_rms quantized per group
//             of 128 to int8: sx_out[g] = absmax / 127, code = value / sx
//             rounded half to even (fp32), bytes in the order int4_a8_unit_dot
//             reads; qs_out[u] = the sum of unit u's 32 codes; returns 1.
// gamma_s: the gain's shared-memory copy from gain_copy_async() (completed by
// this thread before the call), used from the conversion pass on (or null: the
// gain is read from global memory).
// red: shared scratch of 64 floats.  Loads are issued in batches of up to 8
// float4 per thread so that a batch costs one round trip.
//
// Layout: the output is cut into blocks of one weight unit's activations
// (blk_bytes = act_blk_bytes<FMT>(); 0: plain) and the 16-byte chunks inside a
// block are XOR-permuted by the block index, so the lanes of a row slot, which
// read the same chunk of consecutive blocks, hit distinct bank groups.
// swz_offset() gives the permuted byte offset.
// ---------------------------------------------------------------------------
constexpr int kStageBatch = 8;  // float4 loads per thread and staging pass

// The RMSNorm gain is static: the block copies it into shared memory (gs, K
// bf16, 16-byte aligned, K % 8 == 0) as the first cp.async group of every
// thread, before the weight ring's first steps, so that the staging waits on
// the input's round trip only.  The caller then waits with
// cp_async_wait<ring steps issued since>() (every group but the ring's) before
// the staging, whose block barriers publish the copy.
QD_DEV void gain_copy_async(const uint16_t *__restrict__ gamma, int K, uint16_t *gs) {
    if (gamma)
        for (int i = threadIdx.x * 8; i < K; i += blockDim.x * 8) cp_async16(gs + i, gamma + i);
    cp_async_commit();
}

QD_DEV float stage_activations(const float *__restrict__ src, const uint16_t *__restrict__ src_bf16,
                               const uint16_t *__restrict__ gamma, float eps, int K,
                               const float *__restrict__ stats_in, half2 *half_out, float *f32_out,
                               float *red, int blk_bytes = 0, const uint16_t *gamma_s = nullptr,
                               uint8_t *i8_out = nullptr, float *sx_out = nullptr, int *qs_out = nullptr,
                               const long long *__restrict__ src2 = nullptr) {
    constexpr int kBatch = kStageBatch;
    const int tid = threadIdx.x, NT = blockDim.x;
    // src2 (optional): the MLP's pending contribution D in fixed point (delta_to_float),
    // added to src element-wise; the statistics must then be computed here (no stats_in)
    auto load4 = [&](int i) -> float4 {
        if (src_bf16) {
            const uint2 b = *reinterpret_cast<const uint2 *>(src_bf16 + i);
            return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                               __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
        }
        float4 v = __ldcg(reinterpret_cast<const float4 *>(src + i));
        if (src2) {
            const longlong2 d0 = __ldcg(reinterpret_cast<const longlong2 *>(src2 + i));
            const longlong2 d1 = __ldcg(reinterpret_cast<const longlong2 *>(src2 + i + 2));
            v = make_float4(v.x + delta_to_float(d0.x), v.y + delta_to_float(d0.y), v.z + delta_to_float(d1.x),
                            v.w + delta_to_float(d1.y));
        }
        return v;
    };
    bool gs_ok = false;  // the gain's shared-memory copy is visible (after the first barrier)
    auto gain4 = [&](int i) -> float4 {
        if (!gamma) return make_float4(1.f, 1.f, 1.f, 1.f);
        const uint2 g = gs_ok ? *reinterpret_cast<const uint2 *>(gamma_s + i)
                              : __ldg(reinterpret_cast<const uint2 *>(gamma + i));
        return make_float4(__uint_as_float(g.x << 16), __uint_as_float(g.x & 0xFFFF0000u),
                           __uint_as_float(g.y << 16), __uint_as_float(g.y & 0xFFFF0000u));
    };
    const int step = NT * 4;
    float4 v[kBatch];
    // first batch of the input, in flight while the statistics are reduced
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
        const int i = tid * 4 + b * step;
        v[b] = i < K ? load4(i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float ss = 0.f, mx = 0.f;
    if (stats_in) {
        float2 sp[(kStatSlots + 63) / 64];  // blockDim.x >= 64: every pair in one round trip
#pragma unroll
        for (int b = 0; b < (kStatSlots + 63) / 64; ++b) {
            const int c = tid + b * NT;
            sp[b] = c < kStatSlots ? __ldcg(reinterpret_cast<const float2 *>(stats_in) + c) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int b = 0; b < (kStatSlots + 63) / 64; ++b) {
            ss += sp[b].x;
            mx = fmaxf(mx, sp[b].y);
        }
    } else {
        for (int base = 0; base < K; base += kBatch * step) {
            float4 w[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = base + tid * 4 + b * step;
                w[b] = base == 0 ? v[b] : (i < K ? load4(i) : make_float4(0.f, 0.f, 0.f, 0.f));
            }
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = base + tid * 4 + b * step;
                if (i < K) {
                    const float4 g = gain4(i);
                    ss += w[b].x * w[b].x + w[b].y * w[b].y + w[b].z * w[b].z + w[b].w * w[b].w;
                    mx = fmaxf(mx, fmaxf(fmaxf(fabsf(w[b].x * g.x), fabsf(w[b].y * g.y)),
                                         fmaxf(fabsf(w[b].z * g.z), fabsf(w[b].w * g.w))));
                }
            }
        }
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
        float a = lane < (NT + 31) / 32 ? red[lane] : 0.f;
        float b = lane < (NT + 31) / 32 ? red[32 + lane] : 0.f;
        a = warp_sum(a);
        b = warp_max(b);
        if (lane == 0) {
            red[0] = a;
            red[32] = b;
        }
    }
    __syncthreads();
    gs_ok = gamma && gamma_s;
    const float inv = gamma ? rsqrtf(red[0] / (float)K + eps) : 1.f;
    float post = 1.f, pre = inv;
    if (half_out) {
        const float amax = red[32] * inv;
        int e = 0;
        if (amax > 0.f) frexpf(amax, &e);
        pre = ldexpf(inv, -e);
        post = ldexpf(1.f, e);
    }
    for (int base = 0; base < K; base += kBatch * step) {
        if (base > 0) {
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                const int i = base + tid * 4 + b * step;
                if (i < K) v[b] = load4(i);
            }
        }
#pragma unroll
        for (int b = 0; b < kBatch; ++b) {
            const int i = base + tid * 4 + b * step;
            if (i8_out) {
                // int8 per 128-group: a warp's 128 values of this batch are one group
                // (K % 128 == 0, so i < K is warp-uniform); lanes 2m, 2m + 1 hold codes
                // 0-3 and 4-7 of an octet, lanes 8m .. 8m + 7 one 32-code unit
                const bool in = i < K;
                float4 vv = make_float4(0.f, 0.f, 0.f, 0.f);
                if (in) {
                    const float4 g = gain4(i);
                    vv = make_float4(g.x * (v[b].x * pre), g.y * (v[b].y * pre), g.z * (v[b].z * pre),
                                     g.w * (v[b].w * pre));
                }
                const float am = warp_max(fmaxf(fmaxf(fabsf(vv.x), fabsf(vv.y)), fmaxf(fabsf(vv.z), fabsf(vv.w))));
                const float sx = am / 127.f;
                auto qz = [&](float t) -> int {
                    return sx > 0.f ? max(-127, min(127, __float2int_rn(__fdiv_rn(t, sx)))) : 0;
                };
                const int q0 = qz(vv.x), q1 = qz(vv.y), q2 = qz(vv.z), q3 = qz(vv.w);
                const uint32_t p = (uint32_t)(q0 & 255) | ((uint32_t)(q1 & 255) << 8) |
                                   ((uint32_t)(q2 & 255) << 16) | ((uint32_t)(q3 & 255) << 24);
                const uint32_t po = __shfl_xor_sync(0xffffffffu, p, 1);
                int qs = q0 + q1 + q2 + q3;
                qs += __shfl_xor_sync(0xffffffffu, qs, 1);
                qs += __shfl_xor_sync(0xffffffffu, qs, 2);
                qs += __shfl_xor_sync(0xffffffffu, qs, 4);
                const int ln = tid & 31;
                if (in) {
                    if ((ln & 1) == 0) {  // q0 q4 q1 q5 | q2 q6 q3 q7
                        const uint2 wv = make_uint2(prmt(p, po, 0x5140u), prmt(p, po, 0x7362u));
                        *reinterpret_cast<uint2 *>(i8_out + swz_offset((uint32_t)i, blk_bytes)) = wv;
                    }
                    if ((ln & 7) == 0) qs_out[i >> 5] = qs;
                    if (ln == 0) sx_out[i >> 7] = sx;
                }
                continue;
            }
            if (i < K) {
                const float4 g = gain4(i);
                if (half_out) {
                    const uint32_t o = swz_offset((uint32_t)i * 2u, blk_bytes);
                    uint2 hv;
                    hv.x = h2_as_u32(__floats2half2_rn(g.x * (v[b].x * pre), g.y * (v[b].y * pre)));
                    hv.y = h2_as_u32(__floats2half2_rn(g.z * (v[b].z * pre), g.w * (v[b].w * pre)));
                    *reinterpret_cast<uint2 *>(reinterpret_cast<char *>(half_out) + o) = hv;
                } else {
                    const uint32_t o = swz_offset((uint32_t)i * 4u, blk_bytes);
                    *reinterpret_cast<float4 *>(reinterpret_cast<char *>(f32_out) + o) = make_float4(
                        g.x * (v[b].x * pre), g.y * (v[b].y * pre), g.z * (v[b].z * pre), g.w * (v[b].w * pre));
                }
            }
        }
    }
    __syncthreads();
    return post;
}

}  // namespace qd
