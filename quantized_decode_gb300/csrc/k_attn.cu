// k_attn.cu - split-K grouped-query decode attention over the paged bf16 KV cache.
//
// Grid (P, Hkv) in clusters of CS CTAs along x (CS = 8, or 16 where the device
// holds one such cluster per KV head): CTA (p, g) owns KV head g and
// a contiguous run of pages of the T = pos + 1 cached tokens, and serves all
// G = Hq/Hkv query heads of the group from one read of its K/V pages (K and V
// are read once per KV head, not once per query head).
//
// Each warp streams its own pages (the CTA's pages w, w + 8, ...) through a
// two-slot cp.async ring in shared memory, laid out with an XOR swizzle of the
// 16-byte chunks so that ldmatrix reads are conflict-free.  Every page except
// the one being appended is final before the step starts, so the CTA reads the
// position and the page table and issues its first page copies before waiting
// for the QKV kernel; the appended row comes from the bf16 copy that kernel
// writes (kv_new) and replaces its row in shared memory.
//
// Per page the scores S = Q K^T (heads x 16 tokens) and the values O += P V
// are tensor-core contractions (mma.sync m16n8k16, bf16 in, fp32 accumulate).
// Q and P are split into bf16 high and low parts (x = hi + lo, |lo| <= 2^-8 |x|),
// each multiplied separately, so products carry ~16 significant bits while K
// and V are the exact bf16 cache values.  Softmax is online, in base 2.
//
// Partial results merge in three levels, none of which waits on another CTA
// outside its cluster: the 8 warps of a CTA in shared memory; the CS CTAs of a
// cluster through distributed shared memory; the C = P/CS cluster results of a
// KV head by the cluster that arrives last (arrival counter), with the
// log-sum-exp weights e^(m_c - M) / sum_c e^(m_c - M) l_c.  With one cluster
// per KV head (C = 1) the second level writes the output and the third is
// skipped.
#include "attn.cuh"
#include "launch_util.cuh"

namespace qd {

namespace {

using namespace attn;

template <int G, int D, int CS, bool FOLD = false>
__global__ void __launch_bounds__(kNT, 1) k_attn(const __grid_constant__ AttnArgs a) {
    TimelineMark timeline_mark{a.tl};
    extern __shared__ __align__(128) uint16_t smem_raw[];
    uint16_t *smem = align_ring(smem_raw);
    const int g = blockIdx.y;
    auto hook = [&](auto &&) {
        pdl_wait();
        pdl_launch();
        return AttnInputs{a.q + (size_t)g * G * D, a.kv_new ? a.kv_new + (size_t)g * D : nullptr,
                          a.kv_new ? a.kv_new + (size_t)(a.Hkv + g) * D : nullptr};
    };
    attn_cta<G, D, CS, false, false, decltype(hook) &, FOLD>(a, smem, hook);
}


template <int G>
cudaError_t launch_g(const LaunchCfg &lc, const AttnArgs &a) {
    const dim3 grid(a.P, a.Hkv);
    if (a.cs == kCSWide && a.d == 128) {
        if (a.fold) {
            if constexpr (G * 128 % kGroup == 0) {
                if (!allow_wide(k_attn<G, 128, kCSWide, true>)) return cudaErrorInvalidValue;
                return launch_kc(lc, k_attn<G, 128, kCSWide, true>, grid, dim3(kNT), ring_alloc_bytes<128>(), kCSWide,
                                 a);
            }
            return cudaErrorInvalidValue;
        }
        if (!allow_wide(k_attn<G, 128, kCSWide>)) return cudaErrorInvalidValue;
        return launch_kc(lc, k_attn<G, 128, kCSWide>, grid, dim3(kNT), ring_alloc_bytes<128>(), kCSWide, a);
    }
    if (a.fold) return cudaErrorInvalidValue;  // the fold needs one 16-CTA cluster per KV head
    if (a.cs == kCSSmall) {  // several sequences side by side: fewer CTAs per KV head
        if (a.d == 128) return launch_kc(lc, k_attn<G, 128, kCSSmall>, grid, dim3(kNT), ring_alloc_bytes<128>(), kCSSmall, a);
        if (a.d == 64) return launch_kc(lc, k_attn<G, 64, kCSSmall>, grid, dim3(kNT), ring_alloc_bytes<64>(), kCSSmall, a);
        return cudaErrorInvalidValue;
    }
    if (a.cs != 0 && a.cs != kCS) return cudaErrorInvalidValue;
    if (a.d == 128) return launch_kc(lc, k_attn<G, 128, kCS>, grid, dim3(kNT), ring_alloc_bytes<128>(), kCS, a);
    if (a.d == 64) return launch_kc(lc, k_attn<G, 64, kCS>, grid, dim3(kNT), ring_alloc_bytes<64>(), kCS, a);
    return cudaErrorInvalidValue;
}

// Clusters of the kernel that the device holds at once (0 if the query fails).
template <int G, int D, int CS>
int max_clusters_gdc(int Hkv) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, int> cache;  // (device, Hkv) -> clusters
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, Hkv});
    if (it != cache.end()) return it->second;
    const size_t smem = ring_alloc_bytes<D>();
    if (CS > kCS && !allow_wide(k_attn<G, D, CS>)) return 0;
    if (cudaFuncSetAttribute(k_attn<G, D, CS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CS, Hkv);
    cfg.blockDim = dim3(kNT);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = CS;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void *)k_attn<G, D, CS>, &cfg) != cudaSuccess) n = 0;
    cache[{dev, Hkv}] = n;
    return n;
}
template <int G>
int max_clusters_g(int Hkv, int d, int cs) {
    if (cs == kCSWide) return d == 128 ? max_clusters_gdc<G, 128, kCSWide>(Hkv) : 0;
    return d == 128 ? max_clusters_gdc<G, 128, kCS>(Hkv) : max_clusters_gdc<G, 64, kCS>(Hkv);
}
// Clusters of cs CTAs that the device holds at once (0 if unknown).
int max_clusters(int Hq, int Hkv, int d, int cs) {
    if (Hkv < 1 || Hq % Hkv || Hq / Hkv > kMaxGqa || (d != 64 && d != 128)) return 0;
    switch (Hq / Hkv) {
        case 1: return max_clusters_g<1>(Hkv, d, cs);
        case 2: return max_clusters_g<2>(Hkv, d, cs);
        case 3: return max_clusters_g<3>(Hkv, d, cs);
        case 4: return max_clusters_g<4>(Hkv, d, cs);
        case 5: return max_clusters_g<5>(Hkv, d, cs);
        case 6: return max_clusters_g<6>(Hkv, d, cs);
        case 7: return max_clusters_g<7>(Hkv, d, cs);
        default: return max_clusters_g<8>(Hkv, d, cs);
    }
}

// Contexts up to this many pages take one 16-CTA cluster per KV head when it fits.
constexpr int kWideMaxPages = 512;

}  // namespace

int attention_split_multiple() { return kCS; }

int default_splits(int n_sm, int Hq, int Hkv, int d, int max_pages) {
    (void)max_pages;
    int C = n_sm / (kCS * Hkv);
    // every cluster of the grid resident at once: a cluster that has to wait
    // for a free GPC slot starts a second wave and delays the whole step
    const int mc = max_clusters(Hq, Hkv, d, kCS);
    if (mc > 0 && C * Hkv > mc) C = mc / Hkv;
    if (C < 1) C = 1;
    if (C > 32) C = 32;
    return C * kCS;
}

AttnPlan plan_attention(int n_sm, int Hq, int Hkv, int d, int max_pages) {
    // One 16-CTA cluster per KV head: its merge through distributed shared
    // memory gives the final output, with no cross-cluster combine (an atomic
    // arrival and L2 round trips on the step's critical path).  Longer caches
    // keep more, smaller clusters for more SMs streaming K/V.
    if (d == 128 && max_pages <= kWideMaxPages && n_sm >= kCSWide * Hkv &&
        max_clusters(Hq, Hkv, d, kCSWide) >= Hkv)
        return {kCSWide, kCSWide};
    return {default_splits(n_sm, Hq, Hkv, d, max_pages), kCS};
}

namespace {
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled through the runtime's driver entry point (null if unavailable)
EncodeFn tensor_map_encoder() {
    static EncodeFn enc = []() -> EncodeFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeFn>(p);
        return nullptr;
    }();
    return enc;
}
}  // namespace

cudaError_t attention_pool_maps(AttnArgs &a) {
    EncodeFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    if (!a.k_pool || !a.v_pool || ((uintptr_t)a.k_pool & 15) || ((uintptr_t)a.v_pool & 15) || a.n_pages < 1 ||
        a.Hkv < 1 || (a.d != 64 && a.d != 128))
        return cudaErrorInvalidValue;
    const cuuint64_t dims[2] = {(cuuint64_t)a.d, (cuuint64_t)a.n_pages * a.Hkv * kPageTokens};
    const cuuint64_t strides[1] = {(cuuint64_t)a.d * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kPageTokens};
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap *maps[2] = {&a.k_map, &a.v_map};
    const uint16_t *pools[2] = {a.k_pool, a.v_pool};
    for (int i = 0; i < 2; ++i) {
        const CUresult r = enc(maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<uint16_t *>(pools[i]), dims,
                               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

bool attn_fold_ok(int fmt, int Hq, int Hkv, int d, int hidden, const AttnPlan &ap) {
    if (fmt != kFmtInt4 || d != 128 || Hkv < 1 || Hq % Hkv || ap.P != ap.cs || hidden <= 0) return false;
    const int G = Hq / Hkv;
    if (G > 8 || (G * d) % kGroup || hidden % (ap.cs * kWarps) || hidden / ap.cs > 256) return false;
    // the CTA's W_o rows (its KV head's columns), the gathered outputs as fp16 and fp32, the rows'
    // scales, the CTA's merged outputs
    const size_t need = (((size_t)(hidden / ap.cs) * (G * d / 2 + G * d / kGroup * 2) + (size_t)G * d * 6 + 15) & ~(size_t)15) +
                        (size_t)(G * d + ap.cs - 1) / ap.cs * 4;
    return need <= ring_bytes<128>();
}

cudaError_t attn_fold_args(AttnFold &f, const void *wo, const uint16_t *so, long long *out, int Hq, int Hkv, int d,
                           int hidden, const AttnPlan &ap) {
    if (!wo || ((uintptr_t)wo & 15) || !so || !out || !attn_fold_ok(kFmtInt4, Hq, Hkv, d, hidden, ap))
        return cudaErrorInvalidValue;
    EncodeFn enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)Hq * d / 8, (cuuint64_t)hidden};
    const cuuint64_t strides[1] = {(cuuint64_t)Hq * d / 2};
    const cuuint32_t box[2] = {(cuuint32_t)(Hq / Hkv * d / 8), (cuuint32_t)(hidden / ap.cs)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(&f.wo_map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(wo), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    f.so = so;
    f.out = out;
    f.hidden = hidden;
    return cudaSuccess;
}

cudaError_t launch_attention(const LaunchCfg &lc, const AttnArgs &args) {
    const int cs = args.cs == kCSWide ? kCSWide : (args.cs == kCSSmall ? kCSSmall : kCS);
    if (args.P < cs || args.P > 256 || args.P % cs || args.Hkv < 1 || args.Hq % args.Hkv) return cudaErrorInvalidValue;
    if (args.fold && !args.out) return cudaErrorInvalidValue;  // the fold's shapes: attn_fold_args
    AttnArgs a = args;
    const cudaError_t me = attention_pool_maps(a);
    if (me != cudaSuccess) return me;
    switch (a.Hq / a.Hkv) {
        case 1: return launch_g<1>(lc, a);
        case 2: return launch_g<2>(lc, a);
        case 3: return launch_g<3>(lc, a);
        case 4: return launch_g<4>(lc, a);
        case 5: return launch_g<5>(lc, a);
        case 6: return launch_g<6>(lc, a);
        case 7: return launch_g<7>(lc, a);
        case 8: return launch_g<8>(lc, a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qd
