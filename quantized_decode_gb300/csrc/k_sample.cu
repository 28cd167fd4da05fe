// k_sample.cu - temperature / top-k / top-p sampling of the next token on the
// GPU, in place of the greedy argmax ("FlashQwen", run options --temperature,
// --top-k, --top-p, Qwen's recommended 0.6 / 20 / 0.95; naive Qwen engine,
// "Sampler": Top-K draws among the k most probable tokens).
//
// One CTA of 1024 threads over the logits [V] (just written to L2 by the LM head),
// on order-preserving 32-bit keys of the logits, each candidate carried as the
// 64-bit word key << 32 | ~index (so that one descending order is logit
// descending, then index ascending):
//   1. a histogram of the keys' top 12 bits (plain shared-memory atomics) and a
//      suffix scan over it give the bin of the k-th largest key and each bin's
//      first position in the sorted order;
//   2. every key in that bin or above (usually a few hundred) is written into its
//      bin's segment of the candidate array, and ranked by comparison within the
//      segment only -- or, when more than 4096 keys are, the exact slow path:
//      radix select of the k-th largest key (two more 10-bit passes), an ordered
//      compaction (every key above it, then the lowest indices among the keys
//      equal to it), and a bitonic sort;
//   3. in parallel and in fp32: weights exp((l_i - l_0) / T) of the top k, their
//      running sums (a block scan), the top-p cut (the first index whose running
//      sum reaches p of the total), and the draw: the first index whose running
//      sum exceeds u times the prefix's sum, u from SplitMix64 (Steele, Lea &
//      Flood 2014; the published sequential form started at mix(seed), draw
//      number `counter`, top 24 bits * 2^-24).
// The token goes to token_out and, with a state, becomes the next step's input;
// the counter is then the position whose logits are sampled.
#include <climits>

#include "common.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kSampleThreads = 1024;
constexpr int kCand = 4096;   // candidates the fast path collects at most
constexpr int kBatch = 8;     // 16-byte loads in flight per thread in a pass over the logits
constexpr int kRankSeg = 512; // largest bin segment ranked by comparison (else a bitonic sort)

QD_DEV uint32_t order_key(float f) {
    if (f != f) return 0u;  // NaN: below every number
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
QD_DEV float key_value(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

QD_DEV uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Block-wide exclusive scan of one value per thread (1024 threads); returns the
// thread's prefix and writes the total to *total.
QD_DEV int block_exclusive_scan(int v, int *warp_tot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int t = warp_tot[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        warp_tot[lane] = t;  // inclusive over warps
        if (lane == 31) *total = t;
    }
    __syncthreads();
    const int before = (warp ? warp_tot[warp - 1] : 0) + x - v;
    __syncthreads();  // warp_tot is reused by the next scan
    return before;
}

// shared memory (dynamic): bin offsets [4096] u32 | candidates [kCand] u64 | top k [kMaxTopK] u64 | sums [kMaxTopK] f32
constexpr size_t kSampleSmem = 4096 * 4 + kCand * 8 + kMaxTopK * 8 + kMaxTopK * 4;

QD_DEV uint64_t cand_word(uint32_t key, int i) { return ((uint64_t)key << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)i); }
QD_DEV int cand_index(uint64_t c) { return (int)(0xFFFFFFFFu - (uint32_t)c); }

// Bitonic sort of c[0 .. n2) (n2 a power of two) into descending order.
QD_DEV void bitonic_desc(uint64_t *c, int n2) {
    const int tid = threadIdx.x;
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < n2 / 2; t += kSampleThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool desc = (lo & size) == 0;  // this run ends up descending
                const uint64_t x = c[lo], y = c[hi];
                if (desc ? y > x : x > y) {
                    c[lo] = y;
                    c[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(kSampleThreads, 1) k_sample(SampleArgs a) {
    TimelineMark timeline_mark{a.tl};
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t *off = reinterpret_cast<uint32_t *>(smem);                // histogram, then bin offsets
    uint64_t *cand = reinterpret_cast<uint64_t *>(smem + 4096 * 4);
    uint64_t *top = cand + kCand;
    float *cum = reinterpret_cast<float *>(top + kMaxTopK);
    __shared__ uint32_t s_prefix, s_need, s_bin, s_cnt, s_seg;
    __shared__ int s_warp[32], s_total, s_n, s_j;
    __shared__ float s_fw[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int V = a.V, k = a.top_k;

    pdl_wait();
    pdl_launch();
    // the position whose logits are sampled: the draw's counter
    const uint64_t counter = a.st ? (uint64_t)a.st->pos : a.counter;

    // one pass over the logits, f(i, key) for every index: 16-byte loads, kBatch in
    // flight per thread (4-byte loads when the logits are not 16-byte aligned)
    const bool vec = (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0u;
    auto pass = [&](auto &&f) {
        if (vec) {
            const float4 *x4 = reinterpret_cast<const float4 *>(a.logits);
            const int V4 = V >> 2;
            for (int base = 0; base < V4; base += kSampleThreads * kBatch) {
                float4 v[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int i = base + b * kSampleThreads + tid;
                    v[b] = i < V4 ? __ldcg(x4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int i = base + b * kSampleThreads + tid;
                    if (i < V4) {
                        f(4 * i, order_key(v[b].x));
                        f(4 * i + 1, order_key(v[b].y));
                        f(4 * i + 2, order_key(v[b].z));
                        f(4 * i + 3, order_key(v[b].w));
                    }
                }
            }
            for (int i = 4 * V4 + tid; i < V; i += kSampleThreads) f(i, order_key(__ldcg(a.logits + i)));
        } else {
            for (int base = 0; base < V; base += kSampleThreads * kBatch) {
                uint32_t key[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int i = base + b * kSampleThreads + tid;
                    key[b] = i < V ? order_key(__ldcg(a.logits + i)) : 0u;
                }
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    const int i = base + b * kSampleThreads + tid;
                    if (i < V) f(i, key[b]);
                }
            }
        }
    };

    // ---- 1. histogram of the top 12 bits
    for (int b = tid; b < 4096; b += kSampleThreads) off[b] = 0u;
    if (tid == 0) s_seg = 0u;
    __syncthreads();
    pass([&](int, uint32_t key) { atomicAdd(&off[key >> 20], 1u); });
    __syncthreads();
    // suffix scan: thread t owns bins 4095 - 4t - c (c = 0..3), from the top down;
    // off[b] becomes the number of keys in the bins above b (the bin's first position)
    uint32_t h[4];
    int own = 0;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        h[c] = off[4095 - 4 * tid - c];
        own += (int)h[c];
    }
    const int above0 = block_exclusive_scan(own, s_warp, &s_total);
    {
        uint32_t above = (uint32_t)above0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int b = 4095 - 4 * tid - c;
            off[b] = above;
            if (above < (uint32_t)k && above + h[c] >= (uint32_t)k) {  // exactly one bin
                s_bin = (uint32_t)b;
                s_cnt = above + h[c];
            }
            above += h[c];
        }
    }
    __syncthreads();
    const uint32_t bin = s_bin, cnt = s_cnt;
    {  // the largest segment among the candidates' bins
        uint32_t m = 0u;
#pragma unroll
        for (int c = 0; c < 4; ++c)
            if ((uint32_t)(4095 - 4 * tid - c) >= bin) m = max(m, h[c]);
        if (m) atomicMax(&s_seg, m);
    }

    const uint64_t *sorted = top;  // the candidates in descending order, the first k of them
    if (cnt <= (uint32_t)kCand) {
        // ---- 2. the fast path: each key of the bin and above into its bin's segment
        pass([&](int i, uint32_t key) {
            if ((key >> 20) >= bin) cand[atomicAdd(&off[key >> 20], 1u)] = cand_word(key, i);
        });
        __syncthreads();  // off[b] is now the end of bin b's segment, and the start of bin b - 1's
        if (s_seg <= (uint32_t)kRankSeg) {
            // rank = the segment's start + the candidates of the segment ahead of it
            for (int s = tid; s < (int)cnt; s += kSampleThreads) {
                const uint64_t c = cand[s];
                const uint32_t b = (uint32_t)(c >> 52);
                const int st = b == 4095u ? 0 : (int)off[b + 1], en = (int)off[b];
                int r = st;
                for (int j = st; j < en; ++j) r += cand[j] > c;
                if (r < k) top[r] = c;
            }
            __syncthreads();
        } else {
            int n2 = 1;
            while (n2 < (int)cnt) n2 <<= 1;
            for (int s2 = (int)cnt + tid; s2 < n2; s2 += kSampleThreads) cand[s2] = 0ull;
            __syncthreads();
            bitonic_desc(cand, n2);
            sorted = cand;
        }
    } else {
        // ---- 2'. the exact slow path: radix select of the low 20 bits, 10 a pass
        if (tid == 0) {
            s_prefix = bin << 20;
            s_need = (uint32_t)k - off[bin];  // keys of the bin still to take
        }
        uint32_t *hist = reinterpret_cast<uint32_t *>(cand);  // 1024 bins
        uint32_t mask = 0xFFF00000u;
        for (int shift = 10; shift >= 0; shift -= 10) {
            hist[tid] = 0u;
            __syncthreads();
            const uint32_t prefix = s_prefix;
            pass([&](int, uint32_t key) {
                if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 1023u], 1u);
            });
            __syncthreads();
            if (tid == 0) {
                uint32_t need = s_need, acc = 0u;
                int d = 1023;
                for (; d > 0; --d) {
                    if (acc + hist[d] >= need) break;
                    acc += hist[d];
                }
                s_prefix = prefix | ((uint32_t)d << shift);
                s_need = need - acc;  // how many keys equal to the final threshold are taken
            }
            mask |= 1023u << shift;
            __syncthreads();
        }
        const uint32_t thr = s_prefix;
        const int take_eq = (int)s_need;  // >= 1
        const int total_gt = k - take_eq;
        // ordered compaction over tiles of 4 * kSampleThreads consecutive logits (thread t
        // holds 4 consecutive ones, so thread order is index order): the keys above the
        // threshold fill slots 0 .. total_gt - 1, the keys equal to it the slots from
        // total_gt on while they last, both in index order (one scan of the two counts,
        // packed in one word); the next tile is loaded before the current one's scan
        auto load4 = [&](int i0, uint32_t *kk) {
            if (vec && i0 + 3 < V) {
                const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.logits + i0));
                kk[0] = order_key(v.x);
                kk[1] = order_key(v.y);
                kk[2] = order_key(v.z);
                kk[3] = order_key(v.w);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) kk[c] = i0 + c < V ? order_key(__ldcg(a.logits + i0 + c)) : 0u;
            }
        };
        uint32_t cur[4], nxt[4] = {0u, 0u, 0u, 0u};
        load4(4 * tid, cur);
        int gt_base = 0, eq_base = 0;
        for (int t0 = 0; t0 < V; t0 += 4 * kSampleThreads) {
            const int i0 = t0 + 4 * tid;
            if (t0 + 4 * kSampleThreads < V) load4(i0 + 4 * kSampleThreads, nxt);
            int packed = 0;  // keys above << 16 | keys equal (at most 4096 each per tile)
#pragma unroll
            for (int c = 0; c < 4; ++c)
                if (i0 + c < V) packed += cur[c] > thr ? 1 << 16 : (cur[c] == thr ? 1 : 0);
            const int before = block_exclusive_scan(packed, s_warp, &s_total);
            const int tile = s_total;
            int g = gt_base + (before >> 16), e = eq_base + (before & 0xFFFF);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (i0 + c >= V) continue;
                if (cur[c] > thr) {
                    cand[g++] = cand_word(cur[c], i0 + c);
                } else if (cur[c] == thr) {
                    if (e < take_eq) cand[total_gt + e] = cand_word(cur[c], i0 + c);
                    ++e;
                }
            }
            gt_base += tile >> 16;
            eq_base += tile & 0xFFFF;
#pragma unroll
            for (int c = 0; c < 4; ++c) cur[c] = nxt[c];
            if (gt_base >= total_gt && eq_base >= take_eq) break;  // uniform: from the scan's total
        }
        int n2 = 1;
        while (n2 < k) n2 <<= 1;
        for (int s2 = k + tid; s2 < n2; s2 += kSampleThreads) cand[s2] = 0ull;
        __syncthreads();
        bitonic_desc(cand, n2);
        sorted = cand;
    }

    // ---- 3. weights, running sums, the top-p cut and the draw (thread i: candidate i)
    const float l0 = key_value((uint32_t)(sorted[0] >> 32)), t = a.temperature;
    const float w = tid < k ? expf((key_value((uint32_t)(sorted[tid] >> 32)) - l0) / t) : 0.f;
    float x = w;  // inclusive block scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_fw[warp] = x;
    if (tid == 0) {
        s_n = k - 1;
        s_j = INT_MAX;
    }
    __syncthreads();
    if (warp == 0) {
        float y = s_fw[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        s_fw[lane] = y;
    }
    __syncthreads();
    const float run = x + (warp ? s_fw[warp - 1] : 0.f);
    if (tid < k) cum[tid] = run;
    __syncthreads();
    if (a.top_p < 1.f) {
        const float need = a.top_p * cum[k - 1];
        if (tid < k && run >= need) atomicMin(&s_n, tid);
        __syncthreads();
    }
    const int n = s_n;
    const uint64_t xr = sm64_mix(sm64_mix(a.seed) + (counter + 1ull) * 0x9E3779B97F4A7C15ull);
    const float u = (float)(xr >> 40) * 0x1p-24f;
    const float target = u * cum[n];
    if (tid <= n && run > target) atomicMin(&s_j, tid);
    __syncthreads();
    if (tid == 0) {
        const int j = min(s_j, n);
        const int tok = cand_index(sorted[j]);
        *a.token_out = tok;
        if (a.st) {
            a.st->last_token = tok;
            a.st->token = tok;
            if (a.advance) a.st->pos += 1;
        }
    }
}

}  // namespace

cudaError_t launch_sample(const LaunchCfg &lc, const SampleArgs &a) {
    if (!a.logits || !a.token_out || a.V < 1 || a.top_k < 1 || a.top_k > kMaxTopK || a.top_k > a.V ||
        !(a.temperature > 0.f) || !(a.top_p > 0.f) || a.top_p > 1.f)
        return cudaErrorInvalidValue;
    return launch_k(lc, k_sample, dim3(1), dim3(kSampleThreads), kSampleSmem, a);
}

}  // namespace qd
