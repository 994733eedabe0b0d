// Internal interface between the C-ABI entry points and the decode kernels.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

#include "pagedattn.h"

namespace pa {

// Everything a decode launch needs, already validated on the host.
struct DecodeArgs {
    const void* q;                // [batch][num_q_heads][head_dim] of q_dtype
    const void* k_cache;          // [num_blocks][num_kv_heads][block_size][head_dim]
    const void* v_cache;
    const int32_t* block_tables;  // [batch][max_blocks]
    const int32_t* context_lens;  // [batch]
    const int32_t* context_starts;  // [batch] first attended position, or null (all 0)
    void* out;                    // [batch][num_q_heads][head_dim] of out_dtype
    float* part_o;                // [batch][num_q_heads][max_parts][head_dim] (split only)
    float* part_ml;               // [batch][num_q_heads][max_parts][2]: (max, sum) in log2 units
    int32_t* tickets;             // [batch][num_kv_heads * head groups], zero between calls
    int32_t fused_merge;          // 1: the last CTA of a group merges; 0: the merge kernel does
    int32_t balanced_tail;        // 1: the tensor-core kernel shares an item's last chunks among its warps
    int32_t* status;              // device status word or null
    int32_t batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_blocks;
    int32_t group;                // num_q_heads / num_kv_heads
    int32_t partition_size;       // tokens per partition
    int32_t max_parts;            // ceil(max_blocks * block_size / partition_size)
    pa_dtype q_dtype, kv_dtype, out_dtype;
    float scale;                  // softmax scale
    float k_scale, v_scale;       // FP8 dequantisation scales (1 otherwise)
};

// Query heads one CTA serves (a KV head's group is split into chunks of this).
constexpr int kHeadsPerCta = 8;

// CTAs of the tensor-core decode kernel resident per SM (its register budget
// is sized for this many).
#ifndef PA_DECODE_MIN_CTAS
#define PA_DECODE_MIN_CTAS 5
#endif

// CTAs (one warp each) of the warp-per-item decode kernel per SM that its
// register budget is sized for: the residency with FP8 caches (shared
// memory holds 11 with 16-bit caches).
#ifndef PA_DECODE_WARP_MIN_CTAS
#define PA_DECODE_WARP_MIN_CTAS 20
#endif

// Up to this many partitions per sequence the decode kernel merges them itself.
constexpr int kFusedMergeMaxParts = 16;

// Bytes at the front of the decode workspace holding counters that must be
// zero when a call starts (the merge tickets).
size_t decode_counter_bytes(const pa_cache_desc* c, int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                            int32_t partition_size);

// Number of SMs of the current device (cached per device).
int sm_count();

// Host check of a cache descriptor shared by every entry point.
pa_status check_cache_desc(const pa_cache_desc* c);

// Tensor-core kernel: 16-bit or FP8 cache, head_dim 128, 16-bit queries.
bool mma_path_supported(const DecodeArgs& a);
pa_status launch_decode_mma(const DecodeArgs& a, cudaStream_t stream);

// Warp-per-item tensor-core kernel: the same cases as the CTA-per-item
// kernel; chosen when work items are many and long (warp_path_preferred).
pa_status launch_decode_warp(const DecodeArgs& a, cudaStream_t stream);
bool warp_path_preferred(const DecodeArgs& a);

// CUDA-core kernel: every supported combination.
pa_status launch_decode_simt(const DecodeArgs& a, cudaStream_t stream);

// Log-sum-exp merge of the partitions of split sequences.
pa_status launch_decode_reduce(const DecodeArgs& a, cudaStream_t stream);

}  // namespace pa
