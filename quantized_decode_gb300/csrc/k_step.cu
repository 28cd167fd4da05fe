// k_step.cu - the whole decode step as one persistent kernel, one CTA per SM.
//
// Roles.  Warps NCW .. NCW + kStepProducers - 1 produce: lane 0 of each walks
// the step's schedule and takes every kStepProducers-th ring item; for an
// item it waits until the slot is free and issues the TMA copies of what this
// CTA consumes next -- a 3-D box of 4 weight rows x one K-tile (128-byte
// swizzle) plus the cover of the rows' INT4 scales (cp.async.bulk), or K/V
// pages of the paged cache as 128-byte-swizzled 16-row boxes -- completing on
// the slot's `full` mbarrier.  Producers never wait for activations: weights,
// scales and every cached K/V row except the one appended in this step are
// final before the step starts, so the stream runs ahead across phase and
// layer boundaries, limited only by the ring.  Warps 0..NCW-1 consume: per
// phase they wait for the phase's input (a counter that other CTAs raise),
// stage the activations, take the phase's items (item k belongs to warp
// k % NCW: wait `full`, compute, arrive on `empty`) and run the phase's
// epilogue.
//
// Phases per layer (each CTA owns a contiguous share of every phase's rows):
//   QKV  RMSNorm -> Q/K/V GEMV (+bias) -> raw rows; the CTA that completes a
//        head (per-head arrival count) applies the Qwen3 q/k norm and RoPE and
//        writes q, or K/V rounded to bf16 into the page for position pos.
//   ATTN CTA (g, p) of Hkv x P: split p of the cached tokens of KV head g for
//        its G query heads (mma.sync bf16, q and p split into hi/lo parts),
//        then the P CTAs of head g combine the P partials, each one slice of
//        the G*d outputs (log-sum-exp weights).
//   O    o_proj GEMV + residual.
//   GU   RMSNorm -> gate/up GEMV -> SiLU(gate) * up.
//   DOWN down GEMV + residual.
// and LM: final RMSNorm -> LM head GEMV -> logits + argmax; the CTA that
// arrives last reduces the per-CTA maxima, stores the token, advances the
// position and zeroes the step counters for the next step.
//
// Dot products: a lane holds the activations of up to MU 16-byte weight units
// (fp16, scaled per unit by a power of two so |x| < 1) and, for each row
// assigned to its warp, multiplies them with the row's units read from the
// ring (INT4/INT8 codes turned into exact fp16 with lop3/prmt); partial sums
// of 8 rows are combined across the warp with one transposing shuffle tree
// and added into the CTA's per-row results in shared memory.
//
// Every wait is bounded (wait_ns); a wait that runs out records kErrTimeout in
// the device error word, and the CTA leaves at the next phase boundary after
// its producer has seen its outstanding copies land.
#include "gemv.cuh"
#include "launch_util.cuh"
#include "step.h"

namespace qd {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// PTX helpers: mbarriers, TMA, timers, named barriers.
// ---------------------------------------------------------------------------
QD_DEV uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

QD_DEV void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
QD_DEV void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
QD_DEV void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
QD_DEV bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Same, but the thread may sleep (up to `ns`) until the phase completes
// instead of returning at once, so waiting warps do not take issue slots.
QD_DEV bool mbar_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
        : "memory");
    return ok != 0;
}
// L2 policy for data read once per step (weights, cached K/V pages): evicted
// first, so that the stream does not push the kernel's code, parameters and
// activations out of L2.
QD_DEV uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
QD_DEV void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
QD_DEV void tma_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
QD_DEV void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
        "%3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(map), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
QD_DEV uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
QD_DEV int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
QD_DEV int ld_relaxed(const int *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Named barrier 1 over the consumer warps; returns the OR of `pred` over them.
QD_DEV bool cbar_or(int pred, int nthreads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(nthreads)
        : "memory");
    return r != 0;
}
QD_DEV void cbar(int nthreads) { asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory"); }
QD_DEV void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

QD_DEV void ldsm_x4(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
QD_DEV void ldsm_x4_t(const void *p, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
// d += A(16x16; rows 8-15 zero) * B(16x8), bf16 in, fp32 accumulate.
QD_DEV void mma_bf16(float (&d)[2], float &z2, float &z3, uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(z2), "+f"(z3)
        : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}
// x = hi + lo with both bf16 (|lo| <= 2^-8 |x|).
QD_DEV void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

QD_DEV float silu(float a) { return a / (1.f + __expf(-a)); }

// ---------------------------------------------------------------------------
// Schedule shared by producer and consumers.
// ---------------------------------------------------------------------------
QD_DEV void span(int N, int c, int nc, int &r0, int &r1) {
    r0 = (int)((long long)N * c / nc);
    r1 = (int)((long long)N * (c + 1) / nc);
}

// Ring position: the slot and the parity of its current use.
struct RingPos {
    int slot = 0;
    uint32_t par = 0;
    QD_DEV void next(int n) {
        if (++slot == n) {
            slot = 0;
            par ^= 1u;
        }
    }
    QD_DEV void prev(int n) {
        if (--slot < 0) {
            slot = n - 1;
            par ^= 1u;
        }
    }
};

// Row segments of a phase: the QKV rows are q | k | v (three matrices), every
// other phase has one matrix.  Start of segment k = 0..3.
QD_DEV int seg_bound(const StepParams &p, int ph, int k) {
    const int N = p.geo[ph].N;
    if (ph != kPhQkv) return k == 0 ? 0 : N;
    const int b1 = p.Hq * p.d, b2 = b1 + p.Hkv * p.d;
    return k == 0 ? 0 : (k == 1 ? b1 : (k == 2 ? b2 : N));
}

// GEMV ring items of the CTA's rows [r0, r1) of phase ph, in order: blocks
// of up to kStepLines consecutive rows of one segment (gate/up: 2 consecutive
// pairs, lines = gate, gate, up, up), each cut into nt K-tiles.
// f(sg, local, nl, j, t): nl rows (pairs) from row `local` of segment sg, the
// first being the CTA's row j, K-tile t.  Producer and consumers walk this.
template <class Fn>
QD_DEV void for_items(const StepParams &p, int ph, int r0, int r1, Fn &&f) {
    const int nt = p.geo[ph].nt;
    const int rpb = ph == kPhGu ? kStepLines / 2 : kStepLines;
    const int nseg = ph == kPhQkv ? 3 : 1;
    for (int sg = 0; sg < nseg; ++sg) {
        const int b0 = seg_bound(p, ph, sg), b1 = seg_bound(p, ph, sg + 1);
        const int lo = max(r0, b0), hi = min(r1, b1);
        for (int r = lo; r < hi; r += rpb)
            for (int t = 0; t < nt; ++t) f(sg, r - b0, min(rpb, hi - r), r - r0, t);
    }
}

// Codes and scales of segment sg of a phase (gate/up: both matrices).
struct SegMats {
    const uint8_t *wa, *sa, *wb, *sb;
};
QD_DEV SegMats seg_mats(const StepParams &p, const StepLayer &Ly, int ph, int sg) {
    switch (ph) {
        case kPhQkv: return {(const uint8_t *)Ly.w[sg], (const uint8_t *)Ly.s[sg], nullptr, nullptr};
        case kPhO: return {(const uint8_t *)Ly.wo, (const uint8_t *)Ly.so, nullptr, nullptr};
        case kPhGu:
            return {(const uint8_t *)Ly.wg, (const uint8_t *)Ly.sg, (const uint8_t *)Ly.wu, (const uint8_t *)Ly.su};
        case kPhDown: return {(const uint8_t *)Ly.wd, (const uint8_t *)Ly.sd, nullptr, nullptr};
        default: return {(const uint8_t *)p.lm_w, (const uint8_t *)p.lm_scale, nullptr, nullptr};
    }
}

// Tensor maps of segment sg of a phase (gate/up: gate, up).
QD_DEV void seg_maps(const StepParams &p, const StepLayer &Ly, int ph, int sg, const CUtensorMap *&a,
                     const CUtensorMap *&b) {
    b = nullptr;
    switch (ph) {
        case kPhQkv: a = Ly.tm + kMapQ + sg; break;
        case kPhO: a = Ly.tm + kMapO; break;
        case kPhGu:
            a = Ly.tm + kMapGate;
            b = Ly.tm + kMapUp;
            break;
        case kPhDown: a = Ly.tm + kMapDown; break;
        default: a = &p.tm_lm; break;
    }
}

// Byte o of line i of an item's codes (ch = 128-byte chunks per line in the
// box): the 128-byte swizzle permutes the 16-byte units of each segment.
QD_DEV const uint8_t *code_at(const uint8_t *item, int line, int ch, int o) {
    const int seg = line * ch + (o >> 7);
    return item + (seg << 7) + ((((o >> 4) & 7) ^ (seg & 7)) << 4) + (o & 15);
}

// Line i of an item: the matrix row it holds (gate/up: lines 0, 1 gate rows,
// 2, 3 up rows of the same two pairs) and whether it exists (nl rows/pairs).
QD_DEV bool item_line(int ph, int local, int nl, int i, int &row, bool &second) {
    if (ph == kPhGu) {
        second = i >= 2;
        row = local + (i & 1);
        return (i & 1) < nl;
    }
    second = false;
    row = local + i;
    return i < nl;
}
// Bytes of K-tile t of a row, and (INT4) the 16-byte cover of its scales.
QD_DEV int tile_bytes(const StepGeo &g, int t) { return min(g.tk, g.row_bytes - t * g.tk); }

QD_DEV int pages_per_item(int d) { return kStepSlotBytes / (64 * d); }
QD_DEV void attn_split(const StepParams &p, int c, int T, int &g, int &sp, int &pa0, int &pa1) {
    g = c / p.P;
    sp = c % p.P;
    const int n_pg = (T + kPageTokens - 1) / kPageTokens;
    pa0 = (int)((long long)n_pg * sp / p.P);
    pa1 = (int)((long long)n_pg * (sp + 1) / p.P);
}

// Shared-memory carve-up (base aligned to 1024 bytes for the swizzled boxes).
struct Smem {
    uint8_t *ring;
    uint64_t *full, *empty;
    float *res;        // kStepResFloats; the attention phase reuses it
    uint4 *stage;      // staged activations (mma B fragments)
    float *corr;       // per-block offset corrections of the staged activations
    float *red;        // 64 floats of reduction scratch
    int *misc;         // [0] abort, [1..32] finished heads, [33] last-CTA flag,
                       // [34] producers done, [40 + slot] uses of the slot issued
    StepLayer *layers; // copy of the per-layer pointer table
};
constexpr int kMiscProducersDone = 34, kMiscIssued = 40;
static_assert(kMiscIssued + kStepMaxSlots <= 64, "misc words");
QD_HOST_DEV_INLINE size_t smem_bytes(int n_slots, int n_layers) {
    return 1024 + (size_t)n_slots * kStepSlotBytes + (size_t)n_slots * 16 + (size_t)kStepResFloats * 4 +
           kStepStageBytes + 64 * 4 + 64 * 4 + (size_t)n_layers * sizeof(StepLayer);
}
QD_DEV Smem carve(uint8_t *raw, int n_slots) {
    Smem s;
    uint8_t *b = (uint8_t *)(((uintptr_t)raw + 1023) & ~(uintptr_t)1023);
    s.ring = b;
    b += (size_t)n_slots * kStepSlotBytes;
    s.full = (uint64_t *)b;
    s.empty = s.full + n_slots;
    b += (size_t)n_slots * 16;
    s.res = (float *)b;
    b += kStepResFloats * 4;
    s.stage = (uint4 *)b;
    s.corr = (float *)(b + kStepMaxStageK * 2);
    b += kStepStageBytes;
    s.red = (float *)b;
    b += 64 * 4;
    s.misc = (int *)b;
    b += 64 * 4;
    s.layers = (StepLayer *)b;
    return s;
}

// Bounded wait for a device counter to reach `target` (one thread).  Returns
// false (and records the error) when the wait runs out or another CTA failed.
QD_DEV bool wait_counter(const StepParams &p, const int *ctr, int target) {
    const uint64_t t0 = gtimer();
    target += p.test_extra_arrivals;
    for (uint32_t n = 0;; ++n) {
        if (ld_acquire(ctr) >= target) return true;
        if (ld_relaxed(&p.st->err) != kErrNone) return false;
        if ((n & 15) == 15 && gtimer() - t0 > p.counter_wait_ns) {
            atomicCAS(&p.st->err, kErrNone, kErrTimeout);
            return false;
        }
    }
}

// Bounded wait on an mbarrier phase.  `abort` is polled so that a CTA that is
// leaving does not sit out the full bound on every remaining item.
QD_DEV bool wait_mbar(const StepParams &p, uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (;;) {
        if (mbar_wait_sleep(bar, parity, 100000u)) return true;
        if (*abort) return false;
        if (gtimer() - t0 > p.wait_ns) {
            atomicCAS(&p.st->err, kErrNone, kErrTimeout);
            *abort = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Producer.
// ---------------------------------------------------------------------------
template <int DH>
QD_DEV void producer(const StepParams &p, const Smem &s, int pw) {
    // kStepProducers threads (lane 0 of each producer warp) share the copies:
    // producer pw issues the items k with k % kStepProducers == pw of the
    // schedule, so the issue latency of one item overlaps the others'.
    volatile int *abort = s.misc;
    const int c = blockIdx.x, nc = gridDim.x;
    const int T = p.st->pos + 1;
    // Kernel parameters used per item live in registers: every PTX statement
    // below clobbers memory, which would otherwise reload them each time.
    const int n_slots = p.n_slots;
    RingPos rp;          // slot of the current item of the schedule
    int k_item = 0;
    const uint64_t pol = l2_evict_first();
    bool ok = true;
    // Take the schedule's next item: false when it belongs to another
    // producer (or after an abort); else wait until the consumers released
    // the slot's previous use.
    auto claim = [&]() -> bool {
        const bool mine = (k_item++ % kStepProducers) == pw;
        if (mine && ok && !wait_mbar(p, s.empty + rp.slot, rp.par ^ 1u, abort)) ok = false;
        if (!mine || !ok) {
            rp.next(n_slots);
            return false;
        }
        return true;
    };
    auto gemv_items = [&](const StepLayer &Ly, int ph) {
        const StepGeo g = p.geo[ph];
        const int ch = g.tk >> 7;
        int r0, r1;
        span(g.N, c, nc, r0, r1);
        int msg = -1;
        SegMats M{};
        const CUtensorMap *ma = nullptr, *mb = nullptr;
        for_items(p, ph, r0, r1, [&](int sg, int local, int nl, int, int t) {
            if (!claim()) return;
            if (sg != msg) {
                M = seg_mats(p, Ly, ph, sg);
                seg_maps(p, Ly, ph, sg, ma, mb);
                msg = sg;
            }
            uint8_t *dst = s.ring + (size_t)rp.slot * kStepSlotBytes;
            uint64_t *bar = s.full + rp.slot;
            atomicAdd(s.misc + kMiscIssued + rp.slot, 1);
            // codes: one box of 4 rows (gate/up: 2 gate rows, then 2 up rows);
            // INT4 scales: the 16-byte cover of the rows' whole scale rows
            const int lo = (local * g.sr) & ~15, hi = ((local + nl) * g.sr + 15) & ~15;
            const uint32_t cover = g.sr ? (uint32_t)(hi - lo) : 0u;
            mbar_expect_tx(bar, (uint32_t)(kStepLines * ch * 128) + (mb ? 2u : 1u) * cover);
            if (mb) {
                tma_3d(dst, ma, 0, t * ch, local, bar, pol);
                tma_3d(dst + kStepUpOff, mb, 0, t * ch, local, bar, pol);
                if (cover) {
                    bulk_g2s(dst + kStepGuScaleOff, M.sa + lo, cover, bar, pol);
                    bulk_g2s(dst + kStepGuScaleOff + kStepGuScaleSpan, M.sb + lo, cover, bar, pol);
                }
            } else {
                tma_3d(dst, ma, 0, t * ch, local, bar, pol);
                if (cover) bulk_g2s(dst + kStepScaleOff, M.sa + lo, cover, bar, pol);
            }
            rp.next(n_slots);
        });
    };
    auto attn_items = [&](int l) {
        if (c >= p.Hkv * p.P) return;
        int g, sp, pa0, pa1;
        attn_split(p, c, T, g, sp, pa0, pa1);
        const int ppi = pages_per_item(DH);
        for (int k0 = pa0; k0 < pa1; k0 += ppi) {
            const int np = min(ppi, pa1 - k0);
            if (!claim()) continue;
            uint8_t *dst = s.ring + (size_t)rp.slot * kStepSlotBytes;
            uint64_t *bar = s.full + rp.slot;
            atomicAdd(s.misc + kMiscIssued + rp.slot, 1);
            mbar_expect_tx(bar, (uint32_t)(np * 64 * DH));
            for (int k = 0; k < np; ++k) {
                int phys = __ldg(p.page_table + k0 + k);
                if (phys < 0 || phys >= p.n_pages) {
                    atomicCAS(&p.st->err, kErrNone, kErrBadPage);
                    phys = 0;
                }
                const int y = ((l * p.n_pages + phys) * p.Hkv + g) * kPageTokens;
                uint8_t *pgd = dst + (size_t)k * 64 * DH;
#pragma unroll
                for (int hf = 0; hf < DH / 64; ++hf) {
                    tma_2d(pgd + hf * 2048, &p.tm_k, hf * 64, y, bar, pol);
                    tma_2d(pgd + (DH / 64 + hf) * 2048, &p.tm_v, hf * 64, y, bar, pol);
                }
            }
            rp.next(n_slots);
        }
    };
    for (int l = 0; ok && l < p.L; ++l) {
        const StepLayer &Ly = s.layers[l];
        gemv_items(Ly, kPhQkv);
        attn_items(l);
        gemv_items(Ly, kPhO);
        gemv_items(Ly, kPhGu);
        gemv_items(Ly, kPhDown);
    }
    if (ok) gemv_items(s.layers[0], kPhLm);
    // Producer 0 leaves only once every copy issued into the ring has landed
    // (bounded): consumers that gave up early must not leave copies in flight
    // into a CTA that has exited.  It first waits (bounded) until every
    // producer has stopped issuing; then, per slot, the last issued use u - 1
    // is either in flight (the barrier's current phase, waited for) or landed
    // (the phase just before the current one, which the parity wait returns at
    // once).  Uses of a slot land in order, so earlier uses have landed too.
    atomicAdd(s.misc + kMiscProducersDone, 1);
    if (pw == 0) {
        const uint64_t t0 = gtimer();
        while (*(volatile int *)(s.misc + kMiscProducersDone) < kStepProducers && gtimer() - t0 < p.wait_ns) {
        }
        for (int sl = 0; sl < n_slots; ++sl) {
            const int u = *(volatile int *)(s.misc + kMiscIssued + sl);
            if (u == 0) continue;
            const uint32_t par = (uint32_t)(u - 1) & 1u;
            while (!mbar_try_wait(s.full + sl, par) && gtimer() - t0 < p.wait_ns) {
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Consumers: GEMV through mma.sync.
//
// An item (4 row-lines x one K-tile) is owned by one warp.  Its 16 mma rows
// are the 4 lines x 4 K-parts of the tile (part p = blocks [p S, p S + S),
// S = ceil(blocks / 4)); mma row m = part * 4 + line, so thread (gq, tq) feeds
// line gq & 3 of parts gq >> 2 (A rows gq) and 2 + (gq >> 2) (A rows gq + 8),
// and B column n holds the activations of part n.  The k order inside a block
// is permuted the same way on both sides (thread tq takes the block's word /
// quad tq), which leaves every dot product unchanged.  D[m][part(m)] is the
// useful output: thread (gq, 0) holds line gq & 3 of part gq >> 2, thread
// (gq, 1) of part 2 + (gq >> 2); two shuffles sum the parts of a line.
//
// Dequantization folds the code offset into the fp32 accumulator: INT4
// nibbles n = c + 8 become fp16 1024 + n (low pairs) or 1024 + 16 n (high
// pairs, met by activations pre-divided by 16), INT8 bytes c + 128 become
// fp16 1024 + c + 128; the exact per-block sum of activation x offset
// (`corr`) is subtracted in fp32.
// ---------------------------------------------------------------------------
QD_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
QD_DEV void mma_bf16x4(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

QD_DEV float4 ld_act4(const float *src32, const uint16_t *src16, int i) {
    if (src16) {
        const uint2 b = __ldg(reinterpret_cast<const uint2 *>(src16 + i));
        return make_float4(__uint_as_float(b.x << 16), __uint_as_float(b.x & 0xFFFF0000u),
                           __uint_as_float(b.y << 16), __uint_as_float(b.y & 0xFFFF0000u));
    }
    return __ldcg(reinterpret_cast<const float4 *>(src32 + i));
}

// Values per staged chunk: INT4 8 (one 32-bit word of codes), INT8 4, bf16 4.
template <int F>
constexpr int chunk_elems() {
    return F == kFmtInt4 ? 8 : 4;
}
// INT4 staging slot of chunk c (unit u = c / 4, word t = c % 4, group g =
// u / 4): units of odd groups are swapped pairwise so that the four parts of a
// step, whose groups alternate in parity when S is odd, read different banks.
QD_DEV int int4_chunk_slot(int c) {
    const int u = c >> 2, g = u >> 2;
    return ((u ^ (g & 1)) << 2) | (c & 3);
}

// Write chunk c of the (normalized) activations in B-fragment form and return
// its offset sum for the block correction.
template <int F>
QD_DEV float emit_chunk(const Smem &s, int c, const float (&v)[chunk_elems<F>()]) {
    if constexpr (F == kFmtInt4) {
        // positions 2, 3, 6, 7 face the high-nibble pairs (x 16): store them / 16
        const half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2] * 0.0625f, v[3] * 0.0625f);
        const half2 h2 = __floats2half2_rn(v[4], v[5]), h3 = __floats2half2_rn(v[6] * 0.0625f, v[7] * 0.0625f);
        s.stage[int4_chunk_slot(c)] = make_uint4(h2_as_u32(h0), h2_as_u32(h1), h2_as_u32(h2), h2_as_u32(h3));
        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1), f2 = __half22float2(h2), f3 = __half22float2(h3);
        return 1032.f * ((f0.x + f0.y) + (f2.x + f2.y)) + 1152.f * ((f1.x + f1.y) + (f3.x + f3.y));
    } else if constexpr (F == kFmtInt8) {
        const half2 h0 = __floats2half2_rn(v[0], v[1]), h1 = __floats2half2_rn(v[2], v[3]);
        reinterpret_cast<uint2 *>(s.stage)[c] = make_uint2(h2_as_u32(h0), h2_as_u32(h1));
        const float2 f0 = __half22float2(h0), f1 = __half22float2(h1);
        return 1152.f * ((f0.x + f0.y) + (f1.x + f1.y));
    } else {
        uint32_t hi[2], lo[2];
        split2(v[0], v[1], hi[0], lo[0]);
        split2(v[2], v[3], hi[1], lo[1]);
        s.stage[c] = make_uint4(hi[0], hi[1], lo[0], lo[1]);
        return 0.f;
    }
}

// Stage K activations (fp32 src32, or bf16 src16) for the mma GEMV: optional
// RMSNorm with gain gamma, then B-fragment chunks and per-block corrections
// (s.corr[b]: INT4 per 128-code group, INT8 per 16-code block).  Every
// consumer thread calls; ends with a barrier.
template <int F, int NCW>
QD_DEV void stage_mma(const StepParams &p, const Smem &s, const float *src32, const uint16_t *src16,
                      const uint16_t *gamma, int K) {
    constexpr int NCT = NCW * 32;
    constexpr int CE = chunk_elems<F>();
    constexpr int CPB = F == kFmtInt4 ? 16 : 4;  // chunks per correction block
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NC = K / CE;
    auto load = [&](int c, float (&v)[CE]) {
#pragma unroll
        for (int q = 0; q < CE / 4; ++q) {
            const float4 f = ld_act4(src32, src16, c * CE + 4 * q);
            v[4 * q] = f.x;
            v[4 * q + 1] = f.y;
            v[4 * q + 2] = f.z;
            v[4 * q + 3] = f.w;
        }
    };
    // chunk sums -> one correction per block (CPB consecutive lanes)
    auto emit = [&](int c, bool ok, const float (&v)[CE]) {
        float e = ok ? emit_chunk<F>(s, c, v) : 0.f;
        if constexpr (F != kFmtBf16) {
#pragma unroll
            for (int o = CPB / 2; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
            if (ok && (c % CPB) == 0) s.corr[c / CPB] = e;
        }
    };
    if (gamma) {
        // normalized vectors are at most 4096 long: keep them in registers across the reduction
        constexpr int CPT = (4096 / CE + NCT - 1) / NCT;
        float v[CPT][CE];
        float ss = 0.f;
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = tid + k * NCT;
            if (c < NC) {
                load(c, v[k]);
#pragma unroll
                for (int e = 0; e < CE; ++e) ss += v[k][e] * v[k][e];
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) s.red[warp] = ss;
        cbar(NCT);
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) t += s.red[w];
        const float inv = rsqrtf(t / (float)K + p.eps);
#pragma unroll
        for (int k = 0; k < CPT; ++k) {
            const int c = tid + k * NCT;
            const bool ok = c < NC;
            if (ok) {
#pragma unroll
                for (int q = 0; q < CE / 4; ++q) {
                    const uint2 b = __ldg(reinterpret_cast<const uint2 *>(gamma + c * CE + 4 * q));
                    v[k][4 * q] *= __uint_as_float(b.x << 16) * inv;
                    v[k][4 * q + 1] *= __uint_as_float(b.x & 0xFFFF0000u) * inv;
                    v[k][4 * q + 2] *= __uint_as_float(b.y << 16) * inv;
                    v[k][4 * q + 3] *= __uint_as_float(b.y & 0xFFFF0000u) * inv;
                }
            }
            emit(c, ok, v[k]);
        }
    } else {
        for (int base = 0; base < NC; base += NCT) {
            const int c = base + tid;
            const bool ok = c < NC;
            float v[CE];
            if (ok) load(c, v);
            emit(c, ok, v);
        }
    }
    cbar(NCT);
}

// The warp-owned GEMV items of one phase: adds each item's line totals into
// s.res[j * opr + o] (j = row - r0; o = 0 gate / 1 up for gate/up).  Items go
// to the consumer warps round-robin; a warp only waits for and releases its
// own items.  Returns the ring position after the phase.
template <int F, int NCW>
QD_DEV RingPos gemv_mma(const StepParams &p, const Smem &s, int ph, int r0, int r1, RingPos rp) {
    volatile int *abort = s.misc;
    const StepGeo g = p.geo[ph];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, gq = lane >> 2, tq = lane & 3;
    const int line = gq & 3, pa = gq >> 2, pb = 2 + (gq >> 2);
    const int xpart = gq < 4 ? gq : 0;  // B column gq = part gq (columns 4-7 unused)
    const int n_slots = p.n_slots, bb = g.bb;
    const int bpt = g.tk / bb;          // blocks in a full tile
    const int ch = g.tk >> 7;           // 128-byte chunks of a line in the item
    int k = 0;
    for_items(p, ph, r0, r1, [&](int, int local, int nl, int jf, int t) {
        const RingPos q = rp;
        rp.next(n_slots);
        if ((k++ % NCW) != warp) return;
        const bool have = __all_sync(0xffffffffu, wait_mbar(p, s.full + q.slot, q.par, abort));
        const uint8_t *item = s.ring + (size_t)q.slot * kStepSlotBytes;
        // this thread's line inside its box (gate/up: lines 2, 3 are the up box)
        const bool upbox = ph == kPhGu && line >= 2;
        const uint8_t *box = item + (upbox ? kStepUpOff : 0);
        const int bl = upbox ? line - 2 : line;
        int row;
        bool second;
        const bool lvalid = item_line(ph, local, nl, line, row, second);
        const int nb = tile_bytes(g, t) / bb;  // blocks in this tile
        const int S = (nb + 3) >> 2;
        const int b0 = t * bpt;                // first block of the tile in the row
        const int mypart = tq == 0 ? pa : pb;
        float acc = 0.f;
        if (have) {
            if constexpr (F == kFmtInt4) {
                // this line's scales of the tile: its row within the cover, then the tile's groups
                const int first = ph == kPhGu ? (line & 1) : line;
                const uint8_t *cov =
                    item + (ph == kPhGu ? kStepGuScaleOff + (line >= 2 ? kStepGuScaleSpan : 0) : kStepScaleOff);
                const uint16_t *scl = reinterpret_cast<const uint16_t *>(
                                          cov + (local * g.sr - ((local * g.sr) & ~15)) + first * g.sr) + b0;
#pragma unroll 2
                for (int st = 0; st < S; ++st) {
                    const int ba = min(pa * S + st, nb - 1), bq = min(pb * S + st, nb - 1);
                    const int bx = xpart * S + st;
                    const bool xok = bx < nb;
                    const int gx = b0 + min(bx, nb - 1);
                    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t wa = *reinterpret_cast<const uint32_t *>(code_at(box, bl, ch, ba * 64 + j * 16 + tq * 4));
                        const uint32_t wb = *reinterpret_cast<const uint32_t *>(code_at(box, bl, ch, bq * 64 + j * 16 + tq * 4));
                        uint4 xv = s.stage[int4_chunk_slot((gx * 4 + j) * 4 + tq)];
                        if (!xok) xv = make_uint4(0, 0, 0, 0);
                        const uint32_t wa8 = wa >> 8, wb8 = wb >> 8;
                        mma_f16(d, lop3_and_xor(wa, 0x000F000Fu, 0x64086408u), lop3_and_xor(wb, 0x000F000Fu, 0x64086408u),
                                lop3_and_xor(wa, 0x00F000F0u, 0x64806480u), lop3_and_xor(wb, 0x00F000F0u, 0x64806480u),
                                xv.x, xv.y);
                        mma_f16(d, lop3_and_xor(wa8, 0x000F000Fu, 0x64086408u), lop3_and_xor(wb8, 0x000F000Fu, 0x64086408u),
                                lop3_and_xor(wa8, 0x00F000F0u, 0x64806480u), lop3_and_xor(wb8, 0x00F000F0u, 0x64806480u),
                                xv.z, xv.w);
                    }
                    const int bm = mypart * S + st;  // this thread's block (unclamped)
                    const float v = tq == 0 ? (pa ? d[1] : d[0]) : (pb == 3 ? d[3] : d[2]);
                    if (tq < 2 && bm < nb) acc = fmaf(v - s.corr[b0 + bm], bf16_bits_to_float(scl[bm]), acc);
                }
            } else if constexpr (F == kFmtInt8) {
                float d[4] = {0.f, 0.f, 0.f, 0.f}, cor = 0.f;
#pragma unroll 4
                for (int st = 0; st < S; ++st) {
                    const int ba = min(pa * S + st, nb - 1), bq = min(pb * S + st, nb - 1);
                    const int bx = xpart * S + st;
                    uint2 xv = reinterpret_cast<const uint2 *>(s.stage)[(b0 + min(bx, nb - 1)) * 4 + tq];
                    if (bx >= nb) xv = make_uint2(0, 0);
                    const uint32_t wa = *reinterpret_cast<const uint32_t *>(code_at(box, bl, ch, ba * 16 + tq * 4)) ^ 0x80808080u;
                    const uint32_t wb = *reinterpret_cast<const uint32_t *>(code_at(box, bl, ch, bq * 16 + tq * 4)) ^ 0x80808080u;
                    mma_f16(d, prmt(wa, 0x64646464u, 0x4140u), prmt(wb, 0x64646464u, 0x4140u),
                            prmt(wa, 0x64646464u, 0x4342u), prmt(wb, 0x64646464u, 0x4342u), xv.x, xv.y);
                    const int bm = mypart * S + st;
                    if (bm < nb) cor += s.corr[b0 + bm];
                }
                const float v = tq == 0 ? (pa ? d[1] : d[0]) : (pb == 3 ? d[3] : d[2]);
                if (tq < 2) acc = v - cor;
            } else {
                float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                for (int st = 0; st < S; ++st) {
                    const int ba = min(pa * S + st, nb - 1), bq = min(pb * S + st, nb - 1);
                    const int bx = xpart * S + st;
                    uint4 xv = s.stage[(b0 + min(bx, nb - 1)) * 4 + tq];
                    if (bx >= nb) xv = make_uint4(0, 0, 0, 0);
                    const uint2 wa = *reinterpret_cast<const uint2 *>(code_at(box, bl, ch, ba * 32 + tq * 8));
                    const uint2 wb = *reinterpret_cast<const uint2 *>(code_at(box, bl, ch, bq * 32 + tq * 8));
                    mma_bf16x4(d, wa.x, wb.x, wa.y, wb.y, xv.x, xv.y);
                    mma_bf16x4(d, wa.x, wb.x, wa.y, wb.y, xv.z, xv.w);
                }
                const float v = tq == 0 ? (pa ? d[1] : d[0]) : (pb == 3 ? d[3] : d[2]);
                if (tq < 2) acc = v;
            }
        }
        // line total: parts 0/1 (gq, gq + 4) and the tq 0/1 halves
        acc += __shfl_xor_sync(0xffffffffu, acc, 16);
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        if (have && tq == 0 && gq < 4 && lvalid) {
            const int j = jf + (ph == kPhGu ? (line & 1) : line);
            atomicAdd(s.res + (ph == kPhGu ? 2 * j + (second ? 1 : 0) : j), acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(s.empty + q.slot);
    });
    return rp;
}

// ---------------------------------------------------------------------------
// Consumers: phases.
// ---------------------------------------------------------------------------
template <int NCW>
struct Ctx {
    const StepParams &p;
    const Smem &s;
    int c, nc, tid, warp, lane;
    RingPos rp;      // next ring item
    int pos, token;
    bool err;        // this thread saw a failed wait
    volatile int *abort;
    static constexpr int NCT = NCW * 32;

    QD_DEV int *sync_at(int l, int k) const { return p.sync + (size_t)l * kSyncStride + k; }

    // Thread 0 waits for *ctr >= target; all consumers then meet (and agree
    // whether the CTA is leaving).
    QD_DEV bool dep(const int *ctr, int target) {
        if (tid == 0 && ctr && !*abort) {
            if (!wait_counter(p, ctr, target)) *abort = 1;
        }
        return !cbar_or(*abort, NCT);
    }
    // Writes of this CTA are done: make them visible, then raise the counter.
    QD_DEV bool signal(int *ctr, int add) {
        __threadfence();
        const bool fail = cbar_or(*abort, NCT);
        if (tid == 0 && ctr) atomicAdd(ctr, add);
        return !fail;
    }
    QD_DEV void stamp(int k) {
        if (p.prof && c == 0 && tid == 0) p.prof[k] = gtimer();
    }
};

template <int D>
QD_DEV void head_epilogue(const StepParams &p, int l, int head, int pos, int lane) {
    constexpr int M = D / 32;
    float v[M];
    const float *raw = p.raw + (size_t)head * D;
#pragma unroll
    for (int m = 0; m < M; ++m) v[m] = __ldcg(raw + lane + 32 * m);
    const bool is_q = head < p.Hq;
    const bool is_k = !is_q && head < p.Hq + p.Hkv;
    const uint16_t *qg = p.layers[l].q_norm, *kg = p.layers[l].k_norm;
    if ((is_q || is_k) && qg) {
        float ss = 0.f;
#pragma unroll
        for (int m = 0; m < M; ++m) ss += v[m] * v[m];
        ss = warp_sum(ss);
        const float inv = rsqrtf(ss / (float)D + p.eps);
        const uint16_t *gm = is_q ? qg : kg;
#pragma unroll
        for (int m = 0; m < M; ++m) v[m] = bf16_bits_to_float(__ldg(gm + lane + 32 * m)) * (v[m] * inv);
    }
    if (is_q || is_k) {
        const float2 *cs = p.rope_cs + (size_t)pos * (D / 2);
#pragma unroll
        for (int m = 0; m < M / 2; ++m) {
            const float2 cv = __ldg(cs + lane + 32 * m);
            const float x0 = v[m], x1 = v[m + M / 2];
            v[m] = x0 * cv.x - x1 * cv.y;
            v[m + M / 2] = x1 * cv.x + x0 * cv.y;
        }
    }
    if (is_q) {
#pragma unroll
        for (int m = 0; m < M; ++m) p.q[(size_t)head * D + lane + 32 * m] = v[m];
        return;
    }
    const int g = is_k ? head - p.Hq : head - p.Hq - p.Hkv;
    int phys = __ldg(p.page_table + pos / kPageTokens);
    if (phys < 0 || phys >= p.n_pages) {
        if (lane == 0) atomicCAS(&p.st->err, kErrNone, kErrBadPage);
        return;
    }
    uint16_t *dst = (is_k ? p.k_pool : p.v_pool) +
                    ((((size_t)l * p.n_pages + phys) * p.Hkv + g) * kPageTokens + pos % kPageTokens) * D;
#pragma unroll
    for (int m = 0; m < M; ++m) dst[lane + 32 * m] = float_to_bf16_bits(v[m]);
}

template <int DH, int NCW>
QD_DEV bool phase_attn(Ctx<NCW> &x, int l) {
    const StepParams &p = x.p;
    if (x.c >= p.Hkv * p.P) return true;
    constexpr int NKK = DH / 16, NDT = DH / 8;
    constexpr int PB = 64 * DH;  // bytes of one page's K and V boxes
    const int G = p.Hq / p.Hkv;
    const int T = x.pos + 1;
    int g, sp, pa0, pa1;
    attn_split(p, x.c, T, g, sp, pa0, pa1);
    float *s_o = x.s.res;             // [G][DH]
    float *s_m = s_o + 8 * DH;        // [NCW][8]
    float *s_l = s_m + NCW * 8;       // [8]
    for (int i = x.tid; i < 8 * DH + NCW * 8 + 8; i += x.NCT) s_o[i] = i < 8 * DH + NCW * 8 && i >= 8 * DH ? -INFINITY : 0.f;
    if (!x.dep(x.sync_at(l, kSyncHeadsDone), p.Hq + 2 * p.Hkv)) return false;

    const int lane = x.lane, warp = x.warp, gq = lane >> 2, tq = lane & 3;
    uint32_t qh[NKK][2], ql[NKK][2];
#pragma unroll
    for (int kk = 0; kk < NKK; ++kk)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int d0 = kk * 16 + hf * 8 + 2 * tq;
            float q0 = 0.f, q1 = 0.f;
            if (gq < G) {
                const float2 qv = __ldcg(reinterpret_cast<const float2 *>(p.q + (size_t)(g * G + gq) * DH + d0));
                q0 = qv.x;
                q1 = qv.y;
            }
            split2(q0, q1, qh[kk][hf], ql[kk][hf]);
        }
    const float sscale = rsqrtf((float)DH) * kLog2e;
    const int last_pg = (T - 1) / kPageTokens, new_row = (T - 1) % kPageTokens;
    float m = -INFINITY, lsum = 0.f;
    float o[NDT][2];
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) o[dt][0] = o[dt][1] = 0.f;
    float z2 = 0.f, z3 = 0.f;
    const int ppi = pages_per_item(DH);
    int item = 0;
    for (int pa = pa0; pa < pa1; pa += ppi) {
        const int np = min(ppi, pa1 - pa);
        const int slot = x.rp.slot;
        const uint32_t par = x.rp.par;
        x.rp.next(p.n_slots);
        if ((item++ % NCW) != warp) continue;  // each item belongs to one warp
        const bool have = __all_sync(0xffffffffu, wait_mbar(p, x.s.full + slot, par, x.abort));
        for (int k = 0; have && k < np; ++k) {
            const int pg = pa + k;
            uint8_t *kb = x.s.ring + (size_t)slot * kStepSlotBytes + (size_t)k * PB;
            uint8_t *vb = kb + (DH / 64) * 2048;
            auto at = [&](uint8_t *base, int tok, int ch) -> uint8_t * {  // 16-byte chunk ch of row tok
                return base + (ch >> 3) * 2048 + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4);
            };
            if (pg == last_pg) {
                // The appended row, written by this step's QKV phase, and zeros past the sequence.
                int phys = __ldg(p.page_table + pg);
                if (phys < 0 || phys >= p.n_pages) phys = 0;
                const size_t row = ((((size_t)l * p.n_pages + phys) * p.Hkv + g) * kPageTokens + new_row) * DH;
                if (lane < DH / 8) {
                    *reinterpret_cast<uint4 *>(at(kb, new_row, lane)) =
                        __ldcg(reinterpret_cast<const uint4 *>(p.k_pool + row) + lane);
                    *reinterpret_cast<uint4 *>(at(vb, new_row, lane)) =
                        __ldcg(reinterpret_cast<const uint4 *>(p.v_pool + row) + lane);
                }
                for (int cidx = lane; cidx < (kPageTokens - 1 - new_row) * (DH / 8); cidx += 32) {
                    const int tok = new_row + 1 + cidx / (DH / 8), ch = cidx % (DH / 8);
                    *reinterpret_cast<uint4 *>(at(vb, tok, ch)) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async();
                __syncwarp();
            }
            // S = Q K^T for the page's 16 tokens
            float s0[2] = {0.f, 0.f}, s1[2] = {0.f, 0.f};
#pragma unroll
            for (int kk = 0; kk < NKK; ++kk) {
                const int tok = (lane & 7) + ((lane >> 4) << 3);
                const int ch = kk * 2 + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(at(kb, tok, ch), b0, b1, b2, b3);
                mma_bf16(s0, z2, z3, qh[kk][0], qh[kk][1], b0, b1);
                mma_bf16(s0, z2, z3, ql[kk][0], ql[kk][1], b0, b1);
                mma_bf16(s1, z2, z3, qh[kk][0], qh[kk][1], b2, b3);
                mma_bf16(s1, z2, z3, ql[kk][0], ql[kk][1], b2, b3);
            }
            const int base = pg * kPageTokens;
            const float v0 = base + 2 * tq < T ? s0[0] * sscale : -INFINITY;
            const float v1 = base + 2 * tq + 1 < T ? s0[1] * sscale : -INFINITY;
            const float v2 = base + 8 + 2 * tq < T ? s1[0] * sscale : -INFINITY;
            const float v3 = base + 9 + 2 * tq < T ? s1[1] * sscale : -INFINITY;
            float mx = fmaxf(fmaxf(v0, v1), fmaxf(v2, v3));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m, mx);
            const float alpha = exp2f(m - m_new);
            const float p0 = exp2f(v0 - m_new), p1 = exp2f(v1 - m_new);
            const float p2 = exp2f(v2 - m_new), p3 = exp2f(v3 - m_new);
            float ps = (p0 + p1) + (p2 + p3);
            ps += __shfl_xor_sync(0xffffffffu, ps, 1);
            ps += __shfl_xor_sync(0xffffffffu, ps, 2);
            lsum = lsum * alpha + ps;
            m = m_new;
#pragma unroll
            for (int dt = 0; dt < NDT; ++dt) {
                o[dt][0] *= alpha;
                o[dt][1] *= alpha;
            }
            uint32_t ph0, pl0, ph2, pl2;
            split2(p0, p1, ph0, pl0);
            split2(p2, p3, ph2, pl2);
            // O += P V
#pragma unroll
            for (int dp = 0; dp < NDT / 2; ++dp) {
                const int mi = lane >> 3, rr = lane & 7;
                const int tok = rr + (mi & 1) * 8;
                const int ch = dp * 2 + (mi >> 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(at(vb, tok, ch), b0, b1, b2, b3);
                mma_bf16(o[2 * dp], z2, z3, ph0, ph2, b0, b1);
                mma_bf16(o[2 * dp], z2, z3, pl0, pl2, b0, b1);
                mma_bf16(o[2 * dp + 1], z2, z3, ph0, ph2, b2, b3);
                mma_bf16(o[2 * dp + 1], z2, z3, pl0, pl2, b2, b3);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(x.s.empty + slot);
    }
    // ---- merge the warps: common max, then rescaled sums in shared memory
    if (tq == 0 && gq < G) s_m[warp * 8 + gq] = m;
    if (cbar_or(*x.abort, x.NCT)) return false;
    if (gq < G) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NCW; ++w) M = fmaxf(M, s_m[w * 8 + gq]);
        const float f = m == -INFINITY ? 0.f : exp2f(m - M);
        if (f != 0.f) {
#pragma unroll
            for (int dt = 0; dt < NDT; ++dt) {
                atomicAdd(s_o + gq * DH + dt * 8 + 2 * tq, o[dt][0] * f);
                atomicAdd(s_o + gq * DH + dt * 8 + 2 * tq + 1, o[dt][1] * f);
            }
            if (tq == 0) atomicAdd(s_l + gq, lsum * f);
        }
    }
    cbar(x.NCT);
    const size_t slot_base = (size_t)g * p.P + sp;
    for (int idx = x.tid; idx < G * DH; idx += x.NCT) {
        const int h = idx / DH;
        p.part_o[(slot_base * G + h) * DH + idx % DH] = s_o[idx];
        if (idx % DH == 0) {
            float M = -INFINITY;
            for (int w = 0; w < NCW; ++w) M = fmaxf(M, s_m[w * 8 + h]);
            p.part_ml[(slot_base * G + h) * 2] = M;
            p.part_ml[(slot_base * G + h) * 2 + 1] = s_l[h];
        }
    }
    if (!x.signal(x.sync_at(l, kSyncAttnCnt + g), 1)) return false;
    // ---- all P partials of head g are written: combine this CTA's slice
    if (!x.dep(x.sync_at(l, kSyncAttnCnt + g), p.P)) return false;
    const int E = G * DH;
    const int e0 = (int)((long long)E * sp / p.P), e1 = (int)((long long)E * (sp + 1) / p.P);
    const int ne = e1 - e0;
    float *w_ml = x.s.res;             // [P][G] weights, then [G] 1/den
    float *acc = w_ml + p.P * G + 8;   // [ne] sums of the slice
    constexpr int kPer = 4;
    float ov[kPer];
    int oi[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int idx = x.tid + k * x.NCT;
        oi[k] = idx < ne * p.P ? idx : -1;
        ov[k] = 0.f;
        if (oi[k] >= 0) {
            const int pp = idx / ne, e = e0 + idx % ne;
            ov[k] = __ldcg(p.part_o + (((size_t)g * p.P + pp) * G + e / DH) * DH + e % DH);
        }
    }
    for (int idx = x.tid; idx < p.P * G; idx += x.NCT) {
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(p.part_ml) + (size_t)g * p.P * G + idx);
        w_ml[idx] = ml.x;                                  // m, [P][G]
        reinterpret_cast<float *>(x.s.stage)[idx] = ml.y;  // l, [P][G]
    }
    for (int i = x.tid; i < ne; i += x.NCT) acc[i] = 0.f;
    cbar(x.NCT);
    if (x.tid < G) {
        const int h = x.tid;
        float M = -INFINITY;
        for (int pp = 0; pp < p.P; ++pp) M = fmaxf(M, w_ml[pp * G + h]);
        float den = 0.f;
        for (int pp = 0; pp < p.P; ++pp) {
            const float mm = w_ml[pp * G + h];
            const float f = mm == -INFINITY ? 0.f : exp2f(mm - M);
            den = fmaf(f, reinterpret_cast<float *>(x.s.stage)[pp * G + h], den);
            w_ml[pp * G + h] = f;
        }
        w_ml[p.P * G + h] = 1.f / den;
    }
    cbar(x.NCT);
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        if (oi[k] >= 0) {
            const int pp = oi[k] / ne, el = oi[k] % ne, e = e0 + el;
            atomicAdd(acc + el, w_ml[pp * G + e / DH] * ov[k]);
        }
    }
    // partial counts above kPer * NCT per slice are handled by a plain loop
    for (int idx = x.tid + kPer * x.NCT; idx < ne * p.P; idx += x.NCT) {
        const int pp = idx / ne, el = idx % ne, e = e0 + el;
        atomicAdd(acc + el, w_ml[pp * G + e / DH] *
                                __ldcg(p.part_o + (((size_t)g * p.P + pp) * G + e / DH) * DH + e % DH));
    }
    cbar(x.NCT);
    for (int el = x.tid; el < ne; el += x.NCT) {
        const int e = e0 + el;
        p.attn[(size_t)g * G * DH + e] = acc[el] * w_ml[p.P * G + e / DH];
    }
    return x.signal(x.sync_at(l, kSyncAttnDone), 1);
}

// One GEMV phase of a layer (QKV, o_proj, gate/up or down): wait for the
// input, stage it, consume the phase's ring items, run the epilogue and
// signal.  The kernel calls it from a loop that is not unrolled, so its code
// exists once.
template <int WF, int DH, int NCW>
QD_DEV bool layer_gemv(Ctx<NCW> &x, int l, int ph) {
    const StepParams &p = x.p;
    const StepGeo &g = p.geo[ph];
    const StepLayer *Ly = x.s.layers + l;
    const int opr = ph == kPhGu ? 2 : 1;
    int r0, r1;
    span(g.N, x.c, x.nc, r0, r1);
    for (int j = x.tid; j < opr * (r1 - r0); j += x.NCT) x.s.res[j] = 0.f;
    const int *dep = ph == kPhQkv ? (l ? x.sync_at(l - 1, kSyncDDone) : nullptr)
                     : ph == kPhO ? x.sync_at(l, kSyncAttnDone)
                     : ph == kPhGu ? x.sync_at(l, kSyncODone)
                                   : x.sync_at(l, kSyncGuDone);
    if (!x.dep(dep, ph == kPhO ? p.Hkv * p.P : x.nc)) return false;
    const float *src = ph == kPhO ? p.attn : (ph == kPhDown ? p.u : p.x);
    const uint16_t *src16 = ph == kPhQkv && l == 0 ? p.embed + (size_t)x.token * p.h : nullptr;
    const uint16_t *gamma = ph == kPhQkv ? Ly->attn_norm : (ph == kPhGu ? Ly->mlp_norm : nullptr);
    stage_mma<WF, NCW>(p, x.s, src, src16, gamma, g.K);
    x.rp = gemv_mma<WF, NCW>(p, x.s, ph, r0, r1, x.rp);
    if (cbar_or(*x.abort, x.NCT)) return false;
    if (ph == kPhQkv) {
        for (int j = x.tid; j < r1 - r0; j += x.NCT) {
            const int r = r0 + j;
            const int sg = r < seg_bound(p, kPhQkv, 1) ? 0 : (r < seg_bound(p, kPhQkv, 2) ? 1 : 2);
            const int local = r - seg_bound(p, kPhQkv, sg);
            float v = x.s.res[j];
            if (WF == kFmtInt8) v *= __ldg(reinterpret_cast<const float *>(Ly->s[sg]) + local);
            if (Ly->b[sg]) v += bf16_bits_to_float(__ldg(Ly->b[sg] + local));
            p.raw[r] = v;
        }
        __threadfence();
        cbar(x.NCT);
        // Per-head arrival: the CTA that completes a head runs its epilogue.
        const int h_lo = r0 / DH, h_hi = r1 > r0 ? (r1 - 1) / DH : h_lo - 1;
        int *fin = x.s.misc + 1;
        if (x.tid < 32) {
            const int h = h_lo + x.tid;
            int done = 0;
            if (h <= h_hi) {
                const int n = min(r1, (h + 1) * DH) - max(r0, h * DH);
                done = atomicAdd(x.sync_at(l, h), n) + n == DH;
            }
            fin[x.tid] = done;
        }
        cbar(x.NCT);
        for (int t = x.warp; t <= h_hi - h_lo && t < 32; t += NCW) {
            if (!fin[t]) continue;
            __threadfence();
            head_epilogue<DH>(p, l, h_lo + t, x.pos, x.lane);
            __threadfence();
            __syncwarp();
            if (x.lane == 0) atomicAdd(x.sync_at(l, kSyncHeadsDone), 1);
        }
        return true;
    }
    for (int j = x.tid; j < r1 - r0; j += x.NCT) {
        const int r = r0 + j;
        if (ph == kPhGu) {
            float a = x.s.res[2 * j], b = x.s.res[2 * j + 1];
            if (WF == kFmtInt8) {
                a *= __ldg(reinterpret_cast<const float *>(Ly->sg) + r);
                b *= __ldg(reinterpret_cast<const float *>(Ly->su) + r);
            }
            p.u[r] = silu(a) * b;
        } else {
            float v = x.s.res[j];
            if (WF == kFmtInt8) v *= __ldg(reinterpret_cast<const float *>(ph == kPhO ? Ly->so : Ly->sd) + r);
            const float prev = ph == kPhO && l == 0 ? bf16_bits_to_float(__ldg(p.embed + (size_t)x.token * p.h + r))
                                                    : __ldcg(p.x + r);
            p.x[r] = prev + v;
        }
    }
    return x.signal(x.sync_at(l, ph == kPhO ? kSyncODone : (ph == kPhGu ? kSyncGuDone : kSyncDDone)), 1);
}

template <int LMF, int NCW>
QD_DEV void phase_lm(Ctx<NCW> &x, const StepLayer *Ly0) {
    const StepParams &p = x.p;
    const StepGeo &g = p.geo[kPhLm];
    int r0, r1;
    span(g.N, x.c, x.nc, r0, r1);
    for (int j = x.tid; j < r1 - r0; j += x.NCT) x.s.res[j] = 0.f;
    if (!x.dep(x.sync_at(p.L - 1, kSyncDDone), x.nc)) return;
    stage_mma<LMF, NCW>(p, x.s, p.x, nullptr, p.final_norm, g.K);
    x.rp = gemv_mma<LMF, NCW>(p, x.s, kPhLm, r0, r1, x.rp);
    if (cbar_or(*x.abort, x.NCT)) return;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    for (int j = x.tid; j < r1 - r0; j += x.NCT) {
        const int r = r0 + j;
        float v = x.s.res[j];
        if (LMF == kFmtInt8) v *= __ldg(p.lm_scale + r);
        p.logits[r] = v;
        if (v > best || (v == best && r < bi)) {
            best = v;
            bi = r;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) {
            best = ov;
            bi = oi;
        }
    }
    if (x.lane == 0) {
        x.s.red[x.warp] = best;
        reinterpret_cast<int *>(x.s.red)[32 + x.warp] = bi;
    }
    cbar(x.NCT);
    if (x.tid == 0) {
        for (int w = 1; w < NCW; ++w) {
            const float ov = x.s.red[w];
            const int oi = reinterpret_cast<int *>(x.s.red)[32 + w];
            if (ov > best || (ov == best && oi < bi)) {
                best = ov;
                bi = oi;
            }
        }
        p.lm_val[x.c] = best;
        p.lm_idx[x.c] = bi;
        __threadfence();
        const int prev = atomicAdd(p.sync + (size_t)p.L * kSyncStride, 1);
        x.s.misc[33] = prev == x.nc - 1;
    }
    cbar(x.NCT);
    if (!x.s.misc[33]) return;
    __threadfence();
    // Last CTA: global argmax (lowest index on ties), state update, counters reset.
    if (x.warp == 0) {
        float bv = -INFINITY;
        int bix = 0x7fffffff;
        for (int k = x.lane; k < x.nc; k += 32) {
            const float v = __ldcg(p.lm_val + k);
            const int i = __ldcg(p.lm_idx + k);
            if (v > bv || (v == bv && i < bix)) {
                bv = v;
                bix = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bix, o);
            if (ov > bv || (ov == bv && oi < bix)) {
                bv = ov;
                bix = oi;
            }
        }
        if (x.lane == 0) {
            p.st->last_token = bix;
            p.st->token = bix;
            p.st->pos = x.pos + 1;
        }
    }
    for (int i = x.tid; i < p.L * kSyncStride + 1; i += x.NCT) p.sync[i] = 0;
}

// Register split.  The block is 16 warps launched at 128 registers a thread
// (the SM's whole register file): warpgroups 0-2 (the NCW = 12 consumers)
// raise theirs to kConsumerRegs and warpgroup 3 (the producers) lowers its
// own to kProducerRegs; 384 * 152 + 128 * 56 = 65536.  Each SM sub-partition
// runs three consumer warps beside one producer.
constexpr int kLaunchRegs = 128, kConsumerRegs = 152, kProducerRegs = 56;
template <int WF, int LMF, int DH, int NCW>
__global__ void __launch_bounds__((NCW + 4) * 32, 1) k_step(const __grid_constant__ StepParams p) {
    static_assert(NCW == 12 && kStepProducers == 4, "three consumer warpgroups, one producer warpgroup");
    static_assert(NCW * 32 * kConsumerRegs + kStepProducers * 32 * kProducerRegs <= (NCW + 4) * 32 * kLaunchRegs,
                  "register split");
    extern __shared__ uint8_t smem_raw[];
    const Smem s = carve(smem_raw, p.n_slots);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < p.n_slots; ++i) {
            mbar_init(s.full + i, 1);
            mbar_init(s.empty + i, 1);  // each item is released by the one warp that owns it
        }
        s.misc[0] = 0;
        s.misc[kMiscProducersDone] = 0;
        for (int i = 0; i < p.n_slots; ++i) s.misc[kMiscIssued + i] = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    {
        const unsigned long long *src = reinterpret_cast<const unsigned long long *>(p.layers);
        unsigned long long *dst = reinterpret_cast<unsigned long long *>(s.layers);
        const int n = p.L * (int)(sizeof(StepLayer) / 8);
        for (int i = tid; i < n; i += blockDim.x) dst[i] = __ldg(src + i);
    }
    __syncthreads();
    if (warp >= NCW) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
        if (lane == 0) producer<DH>(p, s, warp - NCW);
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
    Ctx<NCW> x{p, s, (int)blockIdx.x, (int)gridDim.x, tid, warp, lane, RingPos{}, 0, 0, false, s.misc};
    x.pos = p.st->pos;
    x.token = p.st->token;
    if (x.token < 0 || x.token >= p.V) {
        if (tid == 0) atomicCAS(&p.st->err, kErrNone, kErrBadToken);
        x.token = 0;
    }
    bool ok = true;
#pragma unroll 1
    for (int l = 0; ok && l < p.L; ++l) {
#pragma unroll 1
        for (int k = 0; ok && k < 5; ++k) {
            x.stamp(5 * l + k);
            if (k == 1) {
                ok = phase_attn<DH, NCW>(x, l);
            } else {
                ok = layer_gemv<WF, DH, NCW>(x, l, k == 0 ? kPhQkv : (k == 2 ? kPhO : (k == 3 ? kPhGu : kPhDown)));
            }
        }
    }
    // the producer may raise `abort` at any time: decide together
    if (!cbar_or(*x.abort, Ctx<NCW>::NCT)) {
        x.stamp(5 * p.L);
        phase_lm<LMF, NCW>(x, s.layers);
        x.stamp(5 * p.L + 1);
    }
}

constexpr int kNcw = 12;

template <int WF, int LMF, int DH>
const void *pick() {
    return (const void *)k_step<WF, LMF, DH, kNcw>;
}

}  // namespace

// ---------------------------------------------------------------------------
// Host: plan, tensor maps, launch.
// ---------------------------------------------------------------------------
bool step_plan(StepParams &p, int weight_fmt, int lm_fmt, int n_sm, int max_smem, StepLaunch &out) {
    if (p.d != 64 && p.d != 128) return false;
    if (p.Hq + 2 * p.Hkv > kSyncMaxHeads || p.Hkv > kSyncMaxKvHeads || p.Hq % p.Hkv) return false;
    const int G = p.Hq / p.Hkv;
    if (G > 8 || n_sm < p.Hkv) return false;
    p.P = n_sm / p.Hkv;
    if (p.P * G + 8 + p.d * G > kStepResFloats || p.P * G * 4 > kStepStageBytes) return false;
    if (n_sm % p.Hkv) return false;  // every CTA takes part in attention
    int n_slots = kStepMaxSlots;
    while (n_slots > 2 && smem_bytes(n_slots, p.L) > (size_t)max_smem) --n_slots;
    if (smem_bytes(n_slots, p.L) > (size_t)max_smem || n_slots < 4) return false;
    p.n_slots = n_slots;
    if (p.inflight < 1) p.inflight = 1;
    if (p.inflight > n_slots) p.inflight = n_slots;
    auto set = [&](int ph, int fmt, int N, int K, int pairs, bool norm) -> bool {
        StepGeo &g = p.geo[ph];
        g.fmt = fmt;
        g.N = N;
        g.K = K;
        (void)norm;
        // mma blocks: INT4 one 128-code group (64 bytes), INT8 16 codes, bf16 16 values
        if (fmt == kFmtInt4 ? K % kGroup : K % 16) return false;
        if (K > kStepMaxStageK || (norm && K > 4096)) return false;
        if (fmt == kFmtBf16 && K * 4 > kStepMaxStageK * 2) return false;  // hi + lo pairs
        if (fmt == kFmtInt8 && K / 16 > 768) return false;                 // corrections per block
        g.row_bytes = fmt == kFmtInt4 ? K / 2 : (fmt == kFmtInt8 ? K : 2 * K);
        g.sr = fmt == kFmtInt4 ? K / 64 : 0;
        g.bb = fmt == kFmtInt4 ? 64 : (fmt == kFmtInt8 ? 16 : 32);
        g.tk = g.row_bytes < kStepTileBytes ? g.row_bytes : kStepTileBytes / g.bb * g.bb;
        g.nt = (g.row_bytes + g.tk - 1) / g.tk;
        // codes: 3-D boxes of 128-byte chunks; INT4 scales: covers of whole scale rows
        if (g.row_bytes % 128 || g.tk % 128) return false;
        const int cover_rows = pairs ? kStepLines / 2 : kStepLines;
        if (g.sr && cover_rows * g.sr + 16 > (pairs ? kStepGuScaleSpan : kStepSlotBytes - kStepScaleOff)) return false;
        // per-CTA rows must fit the result buffer
        const long long rows = ((long long)N + n_sm - 1) / n_sm;
        if (rows * (pairs ? 2 : 1) > kStepResFloats) return false;
        return true;
    };
    const int rq = p.Hq * p.d, rkv = p.Hkv * p.d;
    if (!set(kPhQkv, weight_fmt, rq + 2 * rkv, p.h, 0, true)) return false;
    if (!set(kPhO, weight_fmt, p.h, rq, 0, false)) return false;
    if (!set(kPhGu, weight_fmt, p.F, p.h, 1, true)) return false;
    if (!set(kPhDown, weight_fmt, p.h, p.F, 0, false)) return false;
    if (!set(kPhLm, lm_fmt, p.V, p.h, 0, true)) return false;
    // INT4 scale covers may read up to 15 bytes past a row's scales: every
    // matrix's scale array must end on a 16-byte boundary.
    if (weight_fmt == kFmtInt4) {
        const int Ns[] = {rq, rkv, p.h, p.F};
        const int Ks[] = {p.h, p.h, rq, p.h};
        for (int i = 0; i < 4; ++i)
            if (((long long)Ns[i] * (Ks[i] / 64)) % 16) return false;
        if (((long long)p.h * (p.F / 64)) % 16) return false;
    }
    const void *k = nullptr;
    if (weight_fmt == kFmtInt4 && lm_fmt == kFmtBf16) k = p.d == 128 ? pick<kFmtInt4, kFmtBf16, 128>() : pick<kFmtInt4, kFmtBf16, 64>();
    else if (weight_fmt == kFmtInt8 && lm_fmt == kFmtBf16) k = p.d == 128 ? pick<kFmtInt8, kFmtBf16, 128>() : pick<kFmtInt8, kFmtBf16, 64>();
    else if (weight_fmt == kFmtInt8 && lm_fmt == kFmtInt8) k = p.d == 128 ? pick<kFmtInt8, kFmtInt8, 128>() : pick<kFmtInt8, kFmtInt8, 64>();
    if (!k) return false;
    out.kernel = k;
    out.grid = n_sm;
    out.block = (kNcw + 4) * 32;
    out.smem = smem_bytes(n_slots, p.L);
    return true;
}

cudaError_t step_encode_weight_map(CUtensorMap *map, const void *w, int N, const StepGeo &g, int lines) {
    using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeFn encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
        encode = (EncodeFn)fn;
    }
    if (!w || ((uintptr_t)w & 15) || g.row_bytes % 128 || g.tk % 128 || N < 1) return cudaErrorInvalidValue;
    const cuuint64_t dims[3] = {128, (cuuint64_t)(g.row_bytes / 128), (cuuint64_t)N};
    const cuuint64_t strides[2] = {128, (cuuint64_t)g.row_bytes};
    const cuuint32_t box[3] = {128, (cuuint32_t)(g.tk / 128), (cuuint32_t)lines};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(w), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t step_encode_kv_maps(StepParams &p, size_t total_rows) {
    using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static EncodeFn encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return e != cudaSuccess ? e : cudaErrorNotSupported;
        encode = (EncodeFn)fn;
    }
    if (total_rows >= (1ull << 31)) return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)p.d, (cuuint64_t)total_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)p.d * 2};
    const cuuint32_t box[2] = {64, kPageTokens};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap *maps[2] = {&p.tm_k, &p.tm_v};
    void *bases[2] = {p.k_pool, p.v_pool};
    for (int i = 0; i < 2; ++i) {
        CUresult r = encode(maps[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, bases[i], dims, strides, box, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t step_occupancy(const StepLaunch &sl, int *blocks_per_sm) {
    cudaError_t e = cudaFuncSetAttribute(sl.kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(sl.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl.smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, sl.kernel, sl.block, sl.smem);
    return e;
}

cudaError_t launch_step(const StepLaunch &sl, const StepParams &p, cudaStream_t stream) {
    {
        static std::mutex mu;
        static std::map<std::pair<const void *, int>, size_t> configured;
        int dev = 0;
        cudaError_t ge = cudaGetDevice(&dev);
        if (ge != cudaSuccess) return ge;
        std::lock_guard<std::mutex> lock(mu);
        auto key = std::make_pair(sl.kernel, dev);
        auto it = configured.find(key);
        if (it == configured.end() || it->second < sl.smem) {
            // the whole L1/shared array as shared memory, so that one CTA with
            // its ring fits on every SM (the cooperative launch checks this)
            cudaError_t e = cudaFuncSetAttribute(sl.kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
            e = cudaFuncSetAttribute(sl.kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sl.smem);
            if (e != cudaSuccess) return e;
            configured[key] = sl.smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sl.grid);
    cfg.blockDim = dim3(sl.block);
    cfg.dynamicSmemBytes = sl.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {(void *)&p};
    return cudaLaunchKernelExC(&cfg, sl.kernel, args);
}

}  // namespace qd
