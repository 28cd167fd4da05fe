// launch_util.cuh - cudaLaunchKernelEx with the programmatic-dependent-launch attribute.
#pragma once

#include <cuda_runtime.h>

#include "kernels.h"

namespace qd {

template <typename... KArgs, typename... Args>
cudaError_t launch_k(const LaunchCfg &lc, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                     size_t smem, Args &&...args) {
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = lc.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = lc.pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Largest slot width (lanes per weight row) in {32, 16, 8} dividing the units per row.
inline int pick_lpr(int units) {
    if (units % 32 == 0) return 32;
    if (units % 16 == 0) return 16;
    if (units % 8 == 0) return 8;
    return 0;
}

}  // namespace qd
