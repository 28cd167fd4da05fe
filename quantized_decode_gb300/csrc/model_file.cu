// model_file.cu - the packed model file: write it from host arrays, check its
// header, and create an engine from it (host code; the CUDA runtime for the
// upload).
//
// The pages' runtime keeps the packed weights in one mmap-able binary with a
// 256-byte header that starts with an 8-byte magic, payloads aligned to
// 128-byte L2 lines, and a layout id; the loader refuses a file whose magic or
// layout id is wrong before any weight reaches the GPU, and every tool derives
// the positions of the tensors from the same fixed map instead of reading a
// table ("How To Construct Your Personal LLM Runtime From Scratch", §3 and §4).
// This file keeps those rules with its own magic and header:
//   bytes   0..7   magic "QDECODEW"
//           8..11  format version (1), 12..15 header bytes (256)
//          16..79  llm_config, 16 little-endian 4-byte fields in declaration order
//          80..87  payload offset (256), 88..95 payload bytes
//          96..103 FNV-1a 64 of bytes 0..95; the rest of the header is zero
// then every tensor, each starting on a 128-byte boundary of the file, in the
// order tensor_map() visits them (sizes from the config alone).
#include <cuda_runtime.h>
#include <fcntl.h>
#include <sys/stat.h>
#include <unistd.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "../../include/llm.h"

namespace qd {
void adopt_weight_buffer(llm_t *h, void *dev);  // engine.cu: freed by llm_destroy
}

namespace {

constexpr unsigned char kMagic[8] = {'Q', 'D', 'E', 'C', 'O', 'D', 'E', 'W'};
constexpr uint32_t kVersion = 1;
constexpr uint64_t kHeaderBytes = 256;
constexpr uint64_t kAlign = 128;
constexpr size_t kOffCfg = 16, kOffPayload = 80, kOffPayloadBytes = 88, kOffSum = 96;
static_assert(sizeof(llm_config) == 64, "llm_config is 16 four-byte fields");

uint64_t fnv1a64(const unsigned char *p, size_t n) {
    uint64_t h = 0xcbf29ce484222325ull;
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 0x100000001b3ull;
    }
    return h;
}

// Positive and bounded (a header is only trusted after these checks; the
// bounds are far above any model the engine takes).
bool shape_ok(const llm_config &c) {
    if (c.n_layers <= 0 || c.hidden <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.head_dim <= 0 ||
        c.mlp <= 0 || c.vocab <= 0)
        return false;
    if (c.n_layers > 1024 || c.hidden > 65536 || c.n_q_heads > 1024 || c.n_kv_heads > 1024 || c.head_dim > 1024 ||
        c.mlp > 1 << 20 || c.vocab > 1 << 24)
        return false;
    if (c.weight_format != LLM_FMT_INT4_G128 && c.weight_format != LLM_FMT_INT8_ROW) return false;
    if (c.weight_format == LLM_FMT_INT4_G128 &&
        (c.hidden % 128 || c.mlp % 128 || ((int64_t)c.n_q_heads * c.head_dim) % 128))
        return false;
    return true;
}

int layout_check(const llm_config &c) {
    const int want = c.weight_format == LLM_FMT_INT4_G128 ? LLM_LAYOUT_INT4_VALUESHUFFLE : LLM_LAYOUT_INT8_ROW;
    return c.layout_id == want ? LLM_OK : LLM_ERR_LAYOUT;
}

// Visits every tensor of the model in file order: f(field, bytes), where field
// is the pointer slot of llm_weights / llm_layer_weights that holds it (with
// layers == nullptr every layer visits one scratch struct: sizes only).
template <class F>
void tensor_map(const llm_config &c, llm_weights &w, llm_layer_weights *layers, F &&f) {
    llm_layer_weights scratch{};
    const bool int4 = c.weight_format == LLM_FMT_INT4_G128;
    const int64_t h = c.hidden, qd = (int64_t)c.n_q_heads * c.head_dim, kvd = (int64_t)c.n_kv_heads * c.head_dim;
    const int64_t F_ = c.mlp, V = c.vocab, d = c.head_dim;
    auto wb = [&](int64_t N, int64_t K) { return (uint64_t)(int4 ? N * K / 2 : N * K); };
    auto sb = [&](int64_t N, int64_t K) { return (uint64_t)(int4 ? N * (K / 128) * 2 : N * 4); };
    f(w.embed, (uint64_t)(V * h * 2));
    f(w.final_norm, (uint64_t)(h * 2));
    if (!c.tied_lm_head) {
        if (int4) {
            f(w.lm_head, (uint64_t)(V * h * 2));
        } else {
            f(w.lm_head, (uint64_t)(V * h));
            f(w.lm_scale, (uint64_t)(V * 4));
        }
    }
    for (int l = 0; l < c.n_layers; ++l) {
        llm_layer_weights &L = layers ? layers[l] : scratch;
        f(L.wq, wb(qd, h)), f(L.sq, sb(qd, h));
        if (c.qkv_bias) f(L.bq, (uint64_t)(qd * 2));
        f(L.wk, wb(kvd, h)), f(L.sk, sb(kvd, h));
        if (c.qkv_bias) f(L.bk, (uint64_t)(kvd * 2));
        f(L.wv, wb(kvd, h)), f(L.sv, sb(kvd, h));
        if (c.qkv_bias) f(L.bv, (uint64_t)(kvd * 2));
        f(L.wo, wb(h, qd)), f(L.so, sb(h, qd));
        f(L.wg, wb(F_, h)), f(L.sg, sb(F_, h));
        f(L.wu, wb(F_, h)), f(L.su, sb(F_, h));
        f(L.wd, wb(h, F_)), f(L.sd, sb(h, F_));
        f(L.attn_norm, (uint64_t)(h * 2));
        f(L.mlp_norm, (uint64_t)(h * 2));
        if (c.qk_norm) {
            f(L.q_norm, (uint64_t)(d * 2));
            f(L.k_norm, (uint64_t)(d * 2));
        }
    }
}

uint64_t align_up(uint64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Total file bytes of a model with this configuration.
uint64_t file_bytes(const llm_config &c) {
    llm_weights w{};
    uint64_t off = kHeaderBytes;
    tensor_map(c, w, nullptr, [&](const void *&, uint64_t bytes) { off = align_up(off) + bytes; });
    return off;
}

struct Fd {
    int fd = -1;
    ~Fd() {
        if (fd >= 0) close(fd);
    }
};

bool write_all(int fd, const void *p, uint64_t n) {
    const char *c = static_cast<const char *>(p);
    while (n > 0) {
        const ssize_t k = write(fd, c, n > (1u << 30) ? (1u << 30) : (size_t)n);
        if (k <= 0) return false;
        c += k;
        n -= (uint64_t)k;
    }
    return true;
}

bool read_all(int fd, void *p, uint64_t n, uint64_t at) {
    char *c = static_cast<char *>(p);
    while (n > 0) {
        const ssize_t k = pread(fd, c, n > (1u << 30) ? (1u << 30) : (size_t)n, (off_t)at);
        if (k <= 0) return false;
        c += k;
        n -= (uint64_t)k;
        at += (uint64_t)k;
    }
    return true;
}

// Reads and checks the header of an open file; on success *cfg and
// *payload_bytes describe it.
int read_header(int fd, llm_config *cfg, uint64_t *payload_bytes) {
    unsigned char hdr[kHeaderBytes];
    struct stat st;
    if (fstat(fd, &st) != 0 || (uint64_t)st.st_size < kHeaderBytes || !read_all(fd, hdr, kHeaderBytes, 0))
        return LLM_ERR_FORMAT;
    if (std::memcmp(hdr, kMagic, 8) != 0) return LLM_ERR_FORMAT;
    uint32_t version, hbytes;
    uint64_t poff, pbytes, sum;
    std::memcpy(&version, hdr + 8, 4);
    std::memcpy(&hbytes, hdr + 12, 4);
    std::memcpy(&poff, hdr + kOffPayload, 8);
    std::memcpy(&pbytes, hdr + kOffPayloadBytes, 8);
    std::memcpy(&sum, hdr + kOffSum, 8);
    if (version != kVersion || hbytes != kHeaderBytes || poff != kHeaderBytes || sum != fnv1a64(hdr, kOffSum))
        return LLM_ERR_FORMAT;
    llm_config c;
    std::memcpy(&c, hdr + kOffCfg, sizeof c);
    if (!shape_ok(c)) return LLM_ERR_FORMAT;
    const int lr = layout_check(c);
    if (lr != LLM_OK) return lr;
    const uint64_t total = file_bytes(c);
    if (pbytes != total - kHeaderBytes || (uint64_t)st.st_size < total) return LLM_ERR_FORMAT;
    *cfg = c;
    *payload_bytes = pbytes;
    return LLM_OK;
}

}  // namespace

extern "C" {

int llm_model_file_bytes(const llm_config *cfg, int64_t *bytes) {
    if (!cfg || !bytes || !shape_ok(*cfg)) return LLM_ERR_ARG;
    *bytes = (int64_t)file_bytes(*cfg);
    return LLM_OK;
}

static int model_file_write(const char *path, const llm_config *cfg, const llm_weights *host_weights) {
    if (!path || !cfg || !host_weights || !host_weights->layers || !shape_ok(*cfg)) return LLM_ERR_ARG;
    const int lr = layout_check(*cfg);
    if (lr != LLM_OK) return lr;
    llm_weights w = *host_weights;
    std::vector<llm_layer_weights> layers(host_weights->layers, host_weights->layers + cfg->n_layers);
    bool missing = false;
    tensor_map(*cfg, w, layers.data(), [&](const void *&p, uint64_t) { missing |= p == nullptr; });
    if (missing) return LLM_ERR_ARG;

    unsigned char hdr[kHeaderBytes] = {};
    std::memcpy(hdr, kMagic, 8);
    const uint32_t version = kVersion, hbytes = (uint32_t)kHeaderBytes;
    const uint64_t poff = kHeaderBytes, pbytes = file_bytes(*cfg) - kHeaderBytes;
    std::memcpy(hdr + 8, &version, 4);
    std::memcpy(hdr + 12, &hbytes, 4);
    std::memcpy(hdr + kOffCfg, cfg, sizeof *cfg);
    std::memcpy(hdr + kOffPayload, &poff, 8);
    std::memcpy(hdr + kOffPayloadBytes, &pbytes, 8);
    const uint64_t sum = fnv1a64(hdr, kOffSum);
    std::memcpy(hdr + kOffSum, &sum, 8);

    Fd f;
    f.fd = open(path, O_WRONLY | O_CREAT | O_TRUNC, 0644);
    if (f.fd < 0) return LLM_ERR_IO;
    bool ok = write_all(f.fd, hdr, kHeaderBytes);
    uint64_t off = kHeaderBytes;
    static const unsigned char zeros[kAlign] = {};
    tensor_map(*cfg, w, layers.data(), [&](const void *&p, uint64_t bytes) {
        const uint64_t at = align_up(off);
        ok = ok && write_all(f.fd, zeros, at - off) && write_all(f.fd, p, bytes);
        off = at + bytes;
    });
    ok = ok && fsync(f.fd) == 0;
    return ok ? LLM_OK : LLM_ERR_IO;
}

int llm_model_file_read_config(const char *path, llm_config *cfg_out) {
    if (!path || !cfg_out) return LLM_ERR_ARG;
    Fd f;
    f.fd = open(path, O_RDONLY);
    if (f.fd < 0) return LLM_ERR_IO;
    uint64_t pbytes = 0;
    return read_header(f.fd, cfg_out, &pbytes);
}

static int create_from_file(const char *path, int32_t max_context, void *cuda_stream, llm_t **out) {
    if (!path || !out || max_context < 0) return LLM_ERR_ARG;
    *out = nullptr;
    Fd f;
    f.fd = open(path, O_RDONLY);
    if (f.fd < 0) return LLM_ERR_IO;
    llm_config cfg;
    uint64_t pbytes = 0;
    int rc = read_header(f.fd, &cfg, &pbytes);
    if (rc != LLM_OK) return rc;
    if (max_context > 0) cfg.max_context = max_context;

    // the payload in one device buffer, read in 64 MB chunks through a host buffer
    // (host allocations first: nothing below can throw once the device buffer exists)
    constexpr uint64_t kChunk = 64ull << 20;
    std::vector<char> buf((size_t)(pbytes < kChunk ? pbytes : kChunk));
    std::vector<llm_layer_weights> layers((size_t)cfg.n_layers);
    char *dev = nullptr;
    if (cudaMalloc(&dev, pbytes) != cudaSuccess) return LLM_ERR_CUDA;
    for (uint64_t done = 0; done < pbytes && rc == LLM_OK;) {
        const uint64_t n = pbytes - done < kChunk ? pbytes - done : kChunk;
        if (!read_all(f.fd, buf.data(), n, kHeaderBytes + done)) rc = LLM_ERR_IO;
        else if (cudaMemcpy(dev + done, buf.data(), n, cudaMemcpyHostToDevice) != cudaSuccess) rc = LLM_ERR_CUDA;
        done += n;
    }
    if (rc != LLM_OK) {
        cudaFree(dev);
        return rc;
    }
    llm_weights w{};
    uint64_t off = kHeaderBytes;
    tensor_map(cfg, w, layers.data(), [&](const void *&p, uint64_t bytes) {
        const uint64_t at = align_up(off);
        p = dev + (at - kHeaderBytes);
        off = at + bytes;
    });
    w.layers = layers.data();
    rc = llm_create(&cfg, &w, cuda_stream, out);
    if (rc != LLM_OK) {
        cudaFree(dev);
        return rc;
    }
    qd::adopt_weight_buffer(*out, dev);
    return LLM_OK;
}

// No C++ exception crosses the C ABI (allocation failures become errors).
int llm_model_file_write(const char *path, const llm_config *cfg, const llm_weights *host_weights) {
    try {
        return model_file_write(path, cfg, host_weights);
    } catch (...) {
        return LLM_ERR_IO;
    }
}

int llm_create_from_file(const char *path, int32_t max_context, void *cuda_stream, llm_t **out) {
    if (out) *out = nullptr;
    try {
        return create_from_file(path, max_context, cuda_stream, out);
    } catch (...) {
        return LLM_ERR_IO;
    }
}

}  // extern "C"
