// ops_noalloc.cu - the split-K decode attention entry point that allocates nothing.
//
// Who needs it: callers that may not allocate device memory at the moment they
// call in.  Examples are a serving framework or plugin host that owns every byte
// of device memory through its own fixed pool and forbids cudaMalloc on its
// threads, and latency-critical host paths where cudaMalloc/cudaFree could take a
// driver lock or synchronise the device.  llm_op_attention obtains its scratch
// (per-split partial results and per-KV-head arrival counters) with
// cudaMallocAsync on every call; this variant runs the same kernel with that
// scratch placed in one fixed array of device memory owned by the library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  In host code
// the array's name is only a host-side stand-in, not a device address: the device
// address is obtained once per device with cudaGetSymbolAddress, with that device
// current, on the first call made on that device.  That first call should
// therefore come before any stream capture.  All calls on a device share the one
// array and it keeps the last call's contents; calls whose executions overlap on
// the GPU (different streams, no ordering between them) race on it.  The cached
// address is valid for the life of the device's primary context: the library
// must not be used across a cudaDeviceReset (the module, and with it the array,
// is loaded again at a new address).
#include <mutex>

#include "../../include/llm.h"
#include "../../include/llm_ops.h"
#include "kernels.h"
#include "ops_util.h"

using namespace qd;

namespace {

constexpr size_t kNoAllocScratchBytes = 4u << 20;  // 4 MiB per device
constexpr size_t kCounterBytes = 256;              // arrival counters + error word, zeroed per call
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of g_attn_scratch on the current device (looked up once per device).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return LLM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return LLM_ERR_ARG;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || !p) return LLM_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return LLM_OK;
}

}  // namespace

extern "C" int llm_op_attention_noalloc(const float *q, const void *k_pool, const void *v_pool,
                                        const int32_t *page_table, int32_t n_pool_pages, int32_t T,
                                        int32_t Hq, int32_t Hkv, int32_t d, int32_t n_splits, float *out,
                                        void *stream) {
    if (!q || !k_pool || !v_pool || ((uintptr_t)k_pool & 15) || ((uintptr_t)v_pool & 15) || !page_table ||
        !out || T < 1 || Hkv < 1 || Hq % Hkv || Hq / Hkv > kMaxGqa || (d != 64 && d != 128) ||
        n_splits < 0 || n_splits > 256 || !op_pool_pages_ok(n_pool_pages, Hkv))
        return LLM_ERR_ARG;
    LaunchCfg lc{};
    lc.stream = (cudaStream_t)stream;
    lc.pdl = false;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&lc.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return LLM_ERR_CUDA;
    const int n_pg = (T + kPageTokens - 1) / kPageTokens;
    const int cs = attention_split_multiple();
    const int P = n_splits ? (n_splits + cs - 1) / cs * cs : default_splits(lc.n_sm, Hq, Hkv, d, n_pg);
    if (P > 256) return LLM_ERR_ARG;
    const int G = Hq / Hkv;
    const size_t o_bytes = (size_t)Hkv * P * G * d * 4, ml_bytes = (size_t)Hkv * P * G * 2 * 4;
    // Counters for every KV head plus the error word must fit the zeroed prefix,
    // and the partials the rest of the fixed array.
    if ((size_t)(Hkv + 1) * 4 > kCounterBytes || kCounterBytes + o_bytes + ml_bytes > kNoAllocScratchBytes)
        return LLM_ERR_ARG;
    void *base = nullptr;
    int rc = scratch_address(&base);
    if (rc != LLM_OK) return rc;
    char *scratch = static_cast<char *>(base);
    if (cudaMemsetAsync(scratch, 0, kCounterBytes, lc.stream) != cudaSuccess) return LLM_ERR_CUDA;
    AttnArgs a{};
    a.q = q;
    a.k_pool = (const uint16_t *)k_pool;
    a.v_pool = (const uint16_t *)v_pool;
    a.page_table = page_table;
    a.n_pages = n_pool_pages;
    a.st = nullptr;
    a.T_fixed = T;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.d = d;
    a.P = P;
    a.counter = (int *)scratch;
    a.err = (int *)scratch + Hkv;
    a.part_o = (float *)(scratch + kCounterBytes);
    a.part_ml = (float *)(scratch + kCounterBytes + o_bytes);
    a.out = out;
    if (launch_attention(lc, a) != cudaSuccess) return LLM_ERR_CUDA;
    return op_read_err(a.err, lc.stream);
}
