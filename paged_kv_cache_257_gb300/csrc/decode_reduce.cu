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
#define PA_REDUCE_WARPS 8
#endif
constexpr int kWarps = PA_REDUCE_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kBatch = 8;   // partitions per warp and batch (two batches in flight)
constexpr float kNegInf = -__builtin_huge_valf();

// A batch of partials: kBatch (max, sum) pairs and, per lane, head_dim / 32
// consecutive floats of each partial row (one coalesced row per partition).
template <int N>
struct Batch {
    float2 ml[kBatch];
    float v[kBatch][N];
    // partitions p0, p0 + step, ...; those at or past n_parts read as empty
    __device__ __forceinline__ void load(const float2* mlrow, const float* orow, int p0, int step, int n_parts,
                                         int D) {
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int p = p0 + u * step;
            if (p < n_parts) {
                ml[u] = __ldcg(mlrow + p);
                const float* src = orow + static_cast<int64_t>(p) * D;
                if constexpr (N == 2) {
                    const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
                    v[u][0] = t.x; v[u][1] = t.y;
                } else {
#pragma unroll
                    for (int i = 0; i < N; i += 4) {
                        const float4 t = __ldcg(reinterpret_cast<const float4*>(src + i));
                        v[u][i] = t.x; v[u][i + 1] = t.y; v[u][i + 2] = t.z; v[u][i + 3] = t.w;
                    }
                }
            } else {
                ml[u] = make_float2(kNegInf, 0.f);
#pragma unroll
                for (int i = 0; i < N; ++i) v[u][i] = 0.f;
            }
        }
    }
};

// A running merge (max m, sum l, weighted rows acc) of partials.
template <int N>
struct Running {
    float m = kNegInf, l = 0.f, acc[N];
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = 0.f;
    }
    __device__ __forceinline__ void add(const Batch<N>& b) {
        float mb = kNegInf;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) mb = fmaxf(mb, b.ml[u].x);
        if (mb == kNegInf) return;                      // only empty partitions
        const float mn = fmaxf(m, mb);
        const float s = m == kNegInf ? 0.f : exp2_approx(m - mn);
        l *= s;
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] *= s;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const float w = b.ml[u].x == kNegInf ? 0.f : b.ml[u].y * exp2_approx(b.ml[u].x - mn);
            l += w;
#pragma unroll
            for (int i = 0; i < N; ++i) acc[i] = fmaf(w, b.v[u][i], acc[i]);
        }
        m = mn;
    }
};

// One CTA per (query head, sequence).  Warp w merges partitions w, w +
// kWarps, w + 2 kWarps, ... online (a running maximum, its rows and sum
// rescaled when it grows), kBatch partitions per batch, the next batch's
// loads in flight while the current one is added, so the partials stream
// in without a separate pass for the maximum.  The warps' running merges
// meet in shared memory behind one barrier.
template <int D>
__global__ void __launch_bounds__(kThreads) decode_reduce_kernel(const DecodeArgs a) {
    constexpr int kVec = D / 32;
    __shared__ __align__(16) float s_acc[kWarps][D];
    __shared__ float s_m[kWarps], s_l[kWarps];
    const int hq = blockIdx.x, seq = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();      // the partials come from the previous kernel in the stream
    pdl_trigger();
    const int n_parts = seq_window(a, seq, false).n_parts;
    if (n_parts <= 1) return;
    const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + hq;
    const float2* ml = reinterpret_cast<const float2*>(a.part_ml + row * a.max_parts * 2);
    const float* po = a.part_o + row * a.max_parts * D + lane * kVec;

    Running<kVec> r;
    r.init();
    constexpr int kStride = kWarps * kBatch;   // partitions covered by one batch of every warp
    Batch<kVec> b0, b1;
    b0.load(ml, po, warp, kWarps, n_parts, D);
    for (int p0 = warp; p0 < n_parts; p0 += 2 * kStride) {
        b1.load(ml, po, p0 + kStride, kWarps, n_parts, D);
        r.add(b0);
        if (p0 + kStride >= n_parts) break;
        b0.load(ml, po, p0 + 2 * kStride, kWarps, n_parts, D);
        r.add(b1);
    }

#pragma unroll
    for (int i = 0; i < kVec; ++i) s_acc[warp][lane * kVec + i] = r.acc[i];
    if (lane == 0) {
        s_m[warp] = r.m;
        s_l[warp] = r.l;
    }
    __syncthreads();
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, s_m[w]);
    float coef[kWarps], L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        coef[w] = s_m[w] == kNegInf ? 0.f : exp2_approx(s_m[w] - M);
        L = fmaf(coef[w], s_l[w], L);
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    for (int d = threadIdx.x; d < D; d += kThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t = fmaf(coef[w], s_acc[w][d], t);
        store_out(a.out, row * D + d, t * inv, a.out_dtype);
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
