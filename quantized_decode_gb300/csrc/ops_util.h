// ops_util.h - host helpers shared by the single-kernel entry points (ops.cu,
// ops_noalloc.cu), so that both attention entry points bound the caller's
// pools and report the kernel's error word the same way.
#pragma once

#include <stdint.h>

#include "../../include/llm.h"
#include "kernels.h"

namespace qd {

// The K/V pools hold n_pool_pages pages of [Hkv][16][d]; the attention kernel's
// TMA maps address their rows (page * Hkv * 16 + ...) with int32 coordinates.
inline bool op_pool_pages_ok(int32_t n_pool_pages, int32_t Hkv) {
    return n_pool_pages >= 1 && Hkv >= 1 && (int64_t)n_pool_pages * Hkv * kPageTokens <= INT32_MAX;
}

// Status of a launched kernel from its device error word: waits for `stream`,
// then maps kErrTimeout to LLM_ERR_TIMEOUT and any other set bit to LLM_ERR_DEVICE.
inline int op_read_err(const int *d_err, cudaStream_t stream) {
    int herr = 0;
    if (cudaMemcpyAsync(&herr, d_err, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return LLM_ERR_CUDA;
    if (herr == kErrNone) return LLM_OK;
    return herr == kErrTimeout ? LLM_ERR_TIMEOUT : LLM_ERR_DEVICE;
}

}  // namespace qd
