// k_sample.cu - temperature / top-k / top-p sampling of the next token on the
// GPU, in place of the greedy argmax ("FlashQwen", run options --temperature,
// --top-k, --top-p, Qwen's recommended 0.6 / 20 / 0.95; naive Qwen engine,
// "Sampler": Top-K draws among the k most probable tokens).
//
// One CTA of 1024 threads over the logits [V] (just written to L2 by the LM head):
//   1. radix select of the k-th largest logit on order-preserving 32-bit keys,
//      8 bits a pass from the top (shared-memory histogram, lanes with the same
//      digit add once: __match_any_sync);
//   2. ordered compaction of the k candidates: every key above the threshold,
//      then the lowest indices among the keys equal to it (each thread owns a
//      contiguous index range; block-wide exclusive scans give the offsets);
//   3. bitonic sort of the candidates by (logit descending, index ascending);
//   4. one thread, in that order and in fp32: weights exp((l_i - l_0) / T),
//      running sums, the top-p cut (smallest prefix whose sum reaches p of the
//      total), and the draw: the first index whose running sum exceeds u times
//      the prefix's sum, u from SplitMix64 (Steele, Lea & Flood 2014; the
//      published sequential form started at mix(seed), draw number `counter`,
//      top 24 bits * 2^-24).
// The token goes to token_out and, with a state, becomes the next step's input;
// the counter is then the position whose logits are sampled.
#include <climits>

#include "common.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

constexpr int kSampleThreads = 1024;

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

__global__ void __launch_bounds__(kSampleThreads, 1) k_sample(SampleArgs a) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix, s_need;
    __shared__ int s_warp[32], s_total, s_total2;
    __shared__ uint32_t s_key[kMaxTopK];
    __shared__ int s_idx[kMaxTopK];
    const int tid = threadIdx.x, lane = tid & 31;
    const int V = a.V, k = a.top_k;

    pdl_wait();
    pdl_launch();
    // the position whose logits are sampled: the draw's counter
    const uint64_t counter = a.st ? (uint64_t)a.st->pos : a.counter;

    // ---- 1. the k-th largest key: digit by digit from the top
    if (tid == 0) {
        s_prefix = 0u;
        s_need = (uint32_t)k;
    }
    uint32_t mask = 0u;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += kSampleThreads) hist[b] = 0u;
        __syncthreads();
        const uint32_t prefix = s_prefix;
        for (int base = 0; base < V; base += kSampleThreads) {
            const int i = base + tid;
            uint32_t key = 0u;
            bool in = false;
            if (i < V) {
                key = order_key(__ldcg(a.logits + i));
                in = (key & mask) == prefix;
            }
            const uint32_t digit = in ? (key >> shift) & 255u : 256u;
            const uint32_t peers = __match_any_sync(0xffffffffu, digit);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[digit], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t need = s_need, acc = 0u;
            int d = 255;
            for (; d > 0; --d) {
                if (acc + hist[d] >= need) break;
                acc += hist[d];
            }
            s_prefix = prefix | ((uint32_t)d << shift);
            s_need = need - acc;  // how many keys equal to the final threshold are taken
        }
        mask |= 255u << shift;
        __syncthreads();
    }
    const uint32_t thr = s_prefix;
    const int take_eq = (int)s_need;  // >= 1

    // ---- 2. ordered compaction: thread t owns indices [t * chunk, (t + 1) * chunk)
    const int chunk = (V + kSampleThreads - 1) / kSampleThreads;
    const int i0 = tid * chunk, i1 = min(V, i0 + chunk);
    int n_gt = 0, n_eq = 0;
    for (int i = i0; i < i1; ++i) {
        const uint32_t key = order_key(__ldcg(a.logits + i));
        n_gt += key > thr;
        n_eq += key == thr;
    }
    const int off_gt = block_exclusive_scan(n_gt, s_warp, &s_total);
    const int off_eq = block_exclusive_scan(n_eq, s_warp, &s_total2);
    const int total_gt = s_total;  // == k - take_eq
    {
        int g = off_gt, e = off_eq;
        for (int i = i0; i < i1; ++i) {
            const uint32_t key = order_key(__ldcg(a.logits + i));
            if (key > thr) {
                s_key[g] = key;
                s_idx[g] = i;
                ++g;
            } else if (key == thr) {
                if (e < take_eq) {
                    s_key[total_gt + e] = key;
                    s_idx[total_gt + e] = i;
                }
                ++e;
            }
        }
    }
    // padding up to the sort's power of two
    int n2 = 1;
    while (n2 < k) n2 <<= 1;
    for (int s = k + tid; s < n2; s += kSampleThreads) {
        s_key[s] = 0u;
        s_idx[s] = INT_MAX;
    }
    __syncthreads();

    // ---- 3. bitonic sort: (key descending, index ascending)
    auto before = [&](int x, int y) {  // candidate x goes first
        return s_key[x] > s_key[y] || (s_key[x] == s_key[y] && s_idx[x] < s_idx[y]);
    };
    for (int size = 2; size <= n2; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = tid; t < n2 / 2; t += kSampleThreads) {
                const int lo = 2 * t - (t & (stride - 1));
                const int hi = lo + stride;
                const bool asc = (lo & size) == 0;  // this run ends up in "first-goes-first" order
                if (asc ? before(hi, lo) : before(lo, hi)) {
                    const uint32_t tk = s_key[lo];
                    s_key[lo] = s_key[hi];
                    s_key[hi] = tk;
                    const int ti = s_idx[lo];
                    s_idx[lo] = s_idx[hi];
                    s_idx[hi] = ti;
                }
            }
            __syncthreads();
        }
    }

    // ---- 4. weights, top-p cut and the draw (one thread, in sorted order)
    if (tid == 0) {
        const float l0 = key_value(s_key[0]), t = a.temperature;
        auto weight = [&](int i) { return expf((key_value(s_key[i]) - l0) / t); };
        float total = 0.f;
        for (int i = 0; i < k; ++i) total += weight(i);
        const float need = a.top_p * total;
        float acc = 0.f;
        int n = k - 1;
        if (a.top_p < 1.f) {
            for (int i = 0; i < k; ++i) {
                acc += weight(i);
                if (acc >= need) {
                    n = i;
                    break;
                }
            }
        }
        acc = 0.f;
        float mass = 0.f;
        for (int i = 0; i <= n; ++i) mass += weight(i);
        const uint64_t x = sm64_mix(sm64_mix(a.seed) + (counter + 1ull) * 0x9E3779B97F4A7C15ull);
        const float u = (float)(x >> 40) * 0x1p-24f;
        const float target = u * mass;
        int j = n;
        for (int i = 0; i <= n; ++i) {
            acc += weight(i);
            if (acc > target) {
                j = i;
                break;
            }
        }
        const int tok = s_idx[j];
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
    return launch_k(lc, k_sample, dim3(1), dim3(kSampleThreads), 0, a);
}

}  // namespace qd
