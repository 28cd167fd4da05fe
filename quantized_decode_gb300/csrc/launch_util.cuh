// launch_util.cuh - cudaLaunchKernelEx with the programmatic-dependent-launch attribute.
#pragma once

#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "kernels.h"

namespace qd {

template <typename... KArgs, typename... Args>
cudaError_t launch_kc(const LaunchCfg &lc, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                      size_t smem, int cluster_x, Args &&...args) {
    {
        // Once per kernel and device: every kernel of the step asks for the
        // largest shared-memory carveout, so consecutive kernels never need an
        // SM to drain and re-partition L1/shared memory before the next
        // kernel's CTAs can start beside the running ones (programmatic
        // dependent launch); and opt in to the kernel's dynamic shared memory
        // (static plus dynamic can pass 48 KB even when the dynamic part does not).
        static std::mutex mu;
        static std::map<std::pair<const void *, int>, size_t> configured;
        int dev = 0;
        cudaError_t ge = cudaGetDevice(&dev);
        if (ge != cudaSuccess) return ge;
        std::lock_guard<std::mutex> lock(mu);
        auto key = std::make_pair((const void *)kernel, dev);
        auto it = configured.find(key);
        if (it == configured.end()) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                                 (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) return e;
            it = configured.emplace(key, 0).first;
        }
        if (it->second < smem) {
            cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (e != cudaSuccess) return e;
            it->second = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (lc.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)cluster_x;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Clusters above the portable size (8) need the kernel's opt-in (once per kernel and device).
template <typename K>
bool allow_wide(K kernel) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, bool> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair((const void *)kernel, dev);
    auto it = done.find(key);
    if (it != done.end()) return it->second;
    const bool ok = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
    done[key] = ok;
    return ok;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(const LaunchCfg &lc, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                     size_t smem, Args &&...args) {
    return launch_kc(lc, kernel, grid, block, smem, 1, static_cast<Args &&>(args)...);
}

// Grid plan for a row-tiled GEMV: `tiles` row tiles, each split over `ks` warps
// along K.  Picks tile slots per CTA (tpc, so a CTA has tpc * ks warps, at most
// max_warps) and the grid (at most one CTA per SM) that waste the fewest warp
// slots over the rounds the grid needs, preferring >= 8 warps per SM.
struct GemvPlan {
    int grid, tpc, nw;
};
inline GemvPlan plan_gemv(int tiles, int ks, int n_sm, int max_warps) {
    GemvPlan best{1, 1, ks};
    double best_score = -1.0;
    for (int tpc = 1; tpc * ks <= max_warps; ++tpc) {
        int grid = (tiles + tpc - 1) / tpc;
        if (grid > n_sm) grid = n_sm;
        const int rounds = (tiles + grid * tpc - 1) / (grid * tpc);
        const double eff = (double)tiles / ((double)rounds * grid * tpc);
        const double occ = (double)(tpc * ks) / 8.0;
        const double score = eff * (occ < 1.0 ? occ : 1.0) * ((double)grid / n_sm);
        if (score > best_score + 1e-9) {
            best_score = score;
            best = {grid, tpc, tpc * ks};
        }
    }
    return best;
}

// Largest slot width (lanes per weight row) in {32, 16, 8} dividing the units per row.
inline int pick_lpr(int units) {
    if (units % 32 == 0) return 32;
    if (units % 16 == 0) return 16;
    if (units % 8 == 0) return 8;
    return 0;
}

}  // namespace qd
