// Host-only entry points: version, status names, sizes, slot mapping.
#include <cstdint>
#include <mutex>
#include <vector>

#include <cuda_runtime.h>

#include "decode.h"
#include "pagedattn.h"

namespace pa {

int sm_count() {
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 148;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= static_cast<int>(cache.size())) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

}  // namespace pa

extern "C" {

const char* pa_version(void) { return "pagedattn 0.1.0 (sm_103a)"; }

const char* pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID: return "PA_ERR_INVALID";
        case PA_ERR_OOM: return "PA_ERR_OOM";
        case PA_ERR_RANGE: return "PA_ERR_RANGE";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_FLAG: return "PA_ERR_DEVICE_FLAG";
    }
    return "PA_ERR_UNKNOWN";
}

size_t pa_dtype_size(pa_dtype t) {
    switch (t) {
        case PA_F32: return 4;
        case PA_F16: return 2;
        case PA_BF16: return 2;
        case PA_FP8_E4M3: return 1;
    }
    return 0;
}

// 2 (K and V) x layers x KV heads x head_dim x element bytes: dev.to "Why LLMs
// Run Out of VRAM...", section 2 "The Concrete Math of KV Cache Growth".
uint64_t pa_kv_bytes_per_token(int32_t n_layers, int32_t n_kv_heads, int32_t head_dim, pa_dtype dtype) {
    const uint64_t b = pa_dtype_size(dtype);
    if (n_layers < 0 || n_kv_heads < 0 || head_dim < 0 || b == 0) return 0;
    return 2ull * static_cast<uint64_t>(n_layers) * static_cast<uint64_t>(n_kv_heads) *
           static_cast<uint64_t>(head_dim) * b;
}

// slot = block_tables[seq][pos / block_size] * block_size + pos % block_size:
// section 4 "How the Architecture Works" (block table: logical block ->
// physical block).  All-or-nothing: inputs are checked before any write.
pa_status pa_compute_slot_mapping(const int32_t* block_tables, int32_t batch, int32_t max_blocks,
                                  int32_t block_size, const int32_t* seq_ids, const int32_t* positions,
                                  int32_t num_tokens, int64_t* slots_out) {
    if (num_tokens < 0 || batch < 0 || max_blocks < 0 || block_size <= 0) return PA_ERR_INVALID;
    if (num_tokens == 0) return PA_OK;
    if (!block_tables || !seq_ids || !positions || !slots_out) return PA_ERR_INVALID;
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int32_t s = seq_ids[t], p = positions[t];
        if (s < 0 || s >= batch || p < 0 || p / block_size >= max_blocks) return PA_ERR_RANGE;
    }
    for (int32_t t = 0; t < num_tokens; ++t) {
        const int32_t s = seq_ids[t], p = positions[t];
        const int64_t blk = block_tables[static_cast<int64_t>(s) * max_blocks + p / block_size];
        slots_out[t] = blk * block_size + p % block_size;
    }
    return PA_OK;
}

}  // extern "C"
