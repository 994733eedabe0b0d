// Split-context merge: combine the partition partials of each (sequence,
// query head) into the final output.
//
// Partition p of a sequence left its score maximum m_p and exponent sum l_p
// (both in log2 units of the scaled score) and its normalised output o_p.
// The softmax over the whole context is
//     M = max_p m_p,  w_p = l_p * 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p,
// which is what this kernel computes.  Sequences that fit one partition were
// finished by the decode kernel and are skipped here.  The pages stop at the
// single-pass kernel; this split is the long-context arrangement that keeps
// every SM busy when batch x KV heads is small (hyperinfer.ai "KV cache &
// paged attention deep dive", "Why this matters for long context").
#include "common.cuh"
#include "decode.h"

namespace pa {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 8;   // independent partial loads in flight per lane
constexpr float kNegInf = -__builtin_huge_valf();

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* scratch) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = is_max ? fmaxf(v, o) : v + o;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = scratch[0];
    for (int w = 1; w < kWarps; ++w) r = is_max ? fmaxf(r, scratch[w]) : r + scratch[w];
    __syncthreads();
    return r;
}

// One CTA per (query head, sequence, 32-wide slice of head_dim).  Warp w sums
// partitions w, w+8, ... for the 32 output elements (one per lane, coalesced
// 128-byte rows), kUnroll loads at a time; the 8 warp sums meet in shared memory.
__global__ void __launch_bounds__(kThreads) decode_reduce_kernel(const DecodeArgs a) {
    extern __shared__ float weights[];
    __shared__ float scratch[kWarps];
    __shared__ float sums[kWarps][32];
    const int hq = blockIdx.x, seq = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();      // inputs may come from the previous kernel in the stream
    pdl_trigger();
    int ctx = __ldg(a.context_lens + seq);
    const int cap = a.max_blocks * a.block_size;
    ctx = ctx < 0 ? 0 : (ctx > cap ? cap : ctx);
    const int n_parts = ctx > 0 ? (ctx + a.partition_size - 1) / a.partition_size : 1;
    if (n_parts <= 1) return;
    const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + hq;
    const float* ml = a.part_ml + row * a.max_parts * 2;
    const int d = blockIdx.z * 32 + lane;
    const float* po = a.part_o + row * a.max_parts * a.head_dim + d;

    float M = kNegInf;
    for (int p = threadIdx.x; p < n_parts; p += kThreads) M = fmaxf(M, ml[2 * p]);
    M = block_reduce(M, true, scratch);
    float L = 0.f;
    for (int p = threadIdx.x; p < n_parts; p += kThreads) {
        const float mp = ml[2 * p];
        const float w = mp == kNegInf ? 0.f : ml[2 * p + 1] * exp2_approx(mp - M);
        weights[p] = w;
        L += w;
    }
    L = block_reduce(L, false, scratch);  // its barriers also publish `weights`

    float acc[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) acc[u] = 0.f;
    int p = warp;
    for (; p + (kUnroll - 1) * kWarps < n_parts; p += kUnroll * kWarps) {
        float v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) v[u] = po[static_cast<int64_t>(p + u * kWarps) * a.head_dim];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) acc[u] = fmaf(weights[p + u * kWarps], v[u], acc[u]);
    }
    for (; p < n_parts; p += kWarps) acc[0] = fmaf(weights[p], po[static_cast<int64_t>(p) * a.head_dim], acc[0]);
    float sum = 0.f;
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) sum += acc[u];
    sums[warp][lane] = sum;
    __syncthreads();
    if (warp == 0) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += sums[w][lane];
        store_out(a.out, row * a.head_dim + d, L > 0.f ? t / L : 0.f, a.out_dtype);
    }
}

}  // namespace

pa_status launch_decode_reduce(const DecodeArgs& a, cudaStream_t stream) {
    const int smem = a.max_parts * static_cast<int>(sizeof(float));
    if (smem > 48 * 1024) {
        static cudaError_t err = cudaFuncSetAttribute(decode_reduce_kernel,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 160 * 1024);
        if (err != cudaSuccess) return PA_ERR_CUDA;
    }
    dim3 grid(a.num_q_heads, a.batch, a.head_dim / 32);
    if (launch_pdl(decode_reduce_kernel, grid, dim3(kThreads), smem, stream, a) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

}  // namespace pa
