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
#include "window.cuh"

namespace pa {
namespace {

#ifndef PA_REDUCE_WARPS
#define PA_REDUCE_WARPS 16
#endif
constexpr int kWarps = PA_REDUCE_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kUnroll = 8;   // partitions in flight per warp
constexpr float kNegInf = -__builtin_huge_valf();

// head_dim / 32 consecutive floats of a partial row: one vector load.
template <int N>
struct Slice {
    float v[N];
    __device__ __forceinline__ void load(const float* p) {
        if constexpr (N == 2) {
            const float2 t = __ldcg(reinterpret_cast<const float2*>(p));
            v[0] = t.x; v[1] = t.y;
        } else {
#pragma unroll
            for (int i = 0; i < N; i += 4) {
                const float4 t = __ldcg(reinterpret_cast<const float4*>(p + i));
                v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
            }
        }
    }
};

// One CTA per (query head, sequence).  Every warp takes the maximum of all
// m_p itself, so no barrier precedes the sums; warp w then adds partitions
// w, w+kWarps, ..., kUnroll of them in flight, lane j holding d = j*D/32 ..
// (j+1)*D/32 - 1 of each partial row (one coalesced row per partition).  The
// weights are the same in every lane, so each lane keeps the warp's weight
// sum; the warps' sums meet in shared memory behind one barrier.
template <int D>
__global__ void __launch_bounds__(kThreads) decode_reduce_kernel(const DecodeArgs a) {
    constexpr int kVec = D / 32;
    __shared__ __align__(16) float s_acc[kWarps][D];
    __shared__ float s_l[kWarps];
    const int hq = blockIdx.x, seq = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();      // the partials come from the previous kernel in the stream
    pdl_trigger();
    const int n_parts = seq_window(a, seq, false).n_parts;
    if (n_parts <= 1) return;
    const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + hq;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml + row * a.max_parts * 2);
    const float* po = a.part_o + row * a.max_parts * D + lane * kVec;

    float M = kNegInf;
#pragma unroll 4
    for (int p = lane; p < n_parts; p += 32) M = fmaxf(M, __ldcg(ml + p).x);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));

    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = 0.f;
    float L = 0.f;
    auto add = [&](const float2 mlp, const Slice<kVec>& o) {
        const float w = mlp.x == kNegInf ? 0.f : mlp.y * exp2_approx(mlp.x - M);
        L += w;
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = fmaf(w, o.v[i], acc[i]);
    };
    int p = warp;
    for (; p + (kUnroll - 1) * kWarps < n_parts; p += kUnroll * kWarps) {
        float2 mlp[kUnroll];
        Slice<kVec> o[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            mlp[u] = __ldcg(ml + p + u * kWarps);
            o[u].load(po + static_cast<int64_t>(p + u * kWarps) * D);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) add(mlp[u], o[u]);
    }
    for (; p < n_parts; p += kWarps) {
        Slice<kVec> o;
        o.load(po + static_cast<int64_t>(p) * D);
        add(__ldcg(ml + p), o);
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i) s_acc[warp][lane * kVec + i] = acc[i];
    if (lane == 0) s_l[warp] = L;
    __syncthreads();
    float lt = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) lt += s_l[w];
    for (int d = threadIdx.x; d < D; d += kThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += s_acc[w][d];
        store_out(a.out, row * D + d, lt > 0.f ? t / lt : 0.f, a.out_dtype);
    }
}

}  // namespace

pa_status launch_decode_reduce(const DecodeArgs& a, cudaStream_t stream) {
    const dim3 grid(a.num_q_heads, a.batch);
    cudaError_t err;
    switch (a.head_dim) {
        case 64: err = launch_pdl(decode_reduce_kernel<64>, grid, dim3(kThreads), 0, stream, a); break;
        case 128: err = launch_pdl(decode_reduce_kernel<128>, grid, dim3(kThreads), 0, stream, a); break;
        case 256: err = launch_pdl(decode_reduce_kernel<256>, grid, dim3(kThreads), 0, stream, a); break;
        default: return PA_ERR_UNSUPPORTED;
    }
    return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa
