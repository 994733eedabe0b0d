// Paged decode attention on the CUDA cores, for every supported type mix
// (float32 caches, float32 queries, head_dim 64 / 256, ...).
//
// Same work split and partial format as the tensor-core kernel: one CTA per
// (partition, KV head, sequence) and up to 8 query heads; 4 warps take
// 16-token chunks in turn.  A warp walks its chunk token by token: each lane
// holds head_dim/32 consecutive elements of the token's K and V rows (one
// coalesced row read per warp; the rows of 16 / (head_dim/32) tokens are
// loaded together before the first is used), the dot product with every
// query head is a warp reduction, and the online softmax (running max,
// running sum, rescaled output) is updated in float32, token by token.  Only tokens below the context length are
// read.  dev.to "Why LLMs Run Out of VRAM...", section 4 "The PagedAttention
// CUDA Kernel" (block-table lookup inside the attention loop) and section 1
// (the attention formula).
#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "decode_epilogue.cuh"
#include "window.cuh"

namespace pa {
namespace {

constexpr int kWarps = 4;
constexpr int kChunk = 16;
constexpr float kNegInf = -__builtin_huge_valf();

template <int D>
constexpr int merge_floats() {
    return kWarps * (kHeadsPerCta * (D + 4) + 2 * kHeadsPerCta);
}

__device__ __forceinline__ float load_q(const void* q, int64_t i, pa_dtype t) {
    if (t == PA_F32) return to_float<PA_F32>(q, i);
    if (t == PA_F16) return to_float<PA_F16>(q, i);
    return to_float<PA_BF16>(q, i);
}

template <pa_dtype KV, int D>
__global__ void __launch_bounds__(kWarps * 32) decode_simt_kernel(const DecodeArgs a) {
    constexpr int E = D / 32;  // elements per lane
    constexpr int kTok = 16 / E;   // tokens whose rows are loaded together (2 to 8)
    extern __shared__ float msm[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    const int kvh = blockIdx.y / n_hg, hg = blockIdx.y - kvh * n_hg;
    const int part = blockIdx.x;
    const int bs = a.block_size;

    pdl_wait();      // inputs may come from the previous kernel in the stream
    pdl_trigger();
    const SeqWindow sw = seq_window(a, seq, part == 0 && blockIdx.y == 0 && threadIdx.x == 0);
    const int n_parts = sw.n_parts;
    if (part >= n_parts) return;
    const int tok0 = sw.tok0(part);
    const int tok1 = sw.tok1(part);
    const int h0 = kvh * a.group + hg * kHeadsPerCta;
    const int nh = min(kHeadsPerCta, a.group - hg * kHeadsPerCta);
    const float sc = a.scale * 1.4426950408889634f;
    const float ks = KV == PA_FP8_E4M3 ? a.k_scale : 1.f;
    const float vs = KV == PA_FP8_E4M3 ? a.v_scale : 1.f;

    float qv[kHeadsPerCta][E];
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h) {
        const int64_t base = (static_cast<int64_t>(seq) * a.num_q_heads + h0 + (h < nh ? h : 0)) * D + lane * E;
#pragma unroll
        for (int i = 0; i < E; ++i) qv[h][i] = h < nh ? load_q(a.q, base + i, a.q_dtype) : 0.f;
    }
    float m[kHeadsPerCta], l[kHeadsPerCta], acc[kHeadsPerCta][E];
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h) {
        m[h] = kNegInf;
        l[h] = 0.f;
#pragma unroll
        for (int i = 0; i < E; ++i) acc[h][i] = 0.f;
    }

    const int32_t* bt = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;
    for (int c0 = tok0 + warp * kChunk; c0 < tok1; c0 += kWarps * kChunk) {
        const int c1 = min(tok1, c0 + kChunk);
        const int tl = max(c0, sw.start);
        // the chunk's block ids, one per lane (token c0 + lane), then its K
        // and V rows kTok tokens at a time, all loads of a group in flight
        // before the first is used
        const int my_pb = lane < c1 - c0 ? __ldg(bt + (c0 + lane) / bs) : 0;
        for (int t0 = c0; t0 < c1; t0 += kTok) {
            float kx[kTok][E], vx[kTok][E];
            bool ok[kTok];
#pragma unroll
            for (int u = 0; u < kTok; ++u) {
                const int t = t0 + u;
                const int pb = __shfl_sync(0xffffffffu, my_pb, (t - c0) & 31);
                const bool in = t >= tl && t < c1;
                ok[u] = in && pb >= 0 && pb < a.num_blocks;
                if (in && !ok[u] && lane == 0) raise_flag(a.status, PA_DEVFLAG_BLOCK_RANGE);
                const int64_t row =
                    ok[u] ? ((static_cast<int64_t>(pb) * a.num_kv_heads + kvh) * bs + t % bs) * D + lane * E : 0;
#pragma unroll
                for (int i = 0; i < E; ++i) {
                    kx[u][i] = ok[u] ? to_float<KV>(a.k_cache, row + i) * ks : 0.f;
                    vx[u][i] = ok[u] ? to_float<KV>(a.v_cache, row + i) * vs : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kTok; ++u) {
                if (!ok[u]) continue;
#pragma unroll
                for (int h = 0; h < kHeadsPerCta; ++h) {
                    if (h >= nh) break;
                    float dot = 0.f;
#pragma unroll
                    for (int i = 0; i < E; ++i) dot = fmaf(qv[h][i], kx[u][i], dot);
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
                    const float x = dot * sc;
                    const float mn = fmaxf(m[h], x);
                    const float al = exp2_approx(m[h] - mn);
                    const float p = exp2_approx(x - mn);
                    l[h] = l[h] * al + p;
#pragma unroll
                    for (int i = 0; i < E; ++i) acc[h][i] = fmaf(p, vx[u][i], acc[h][i] * al);
                    m[h] = mn;
                }
            }
        }
    }

    // merge the 4 warps' states in shared memory
    float* mbuf = msm;
    float* mm = mbuf + kWarps * kHeadsPerCta * (D + 4);
    float* ml = mm + kWarps * kHeadsPerCta;
#pragma unroll
    for (int h = 0; h < kHeadsPerCta; ++h) {
#pragma unroll
        for (int i = 0; i < E; ++i) mbuf[(warp * kHeadsPerCta + h) * (D + 4) + lane * E + i] = acc[h][i];
        if (lane == 0) {
            mm[warp * kHeadsPerCta + h] = m[h];
            ml[warp * kHeadsPerCta + h] = l[h];
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
        const int h = idx / D, d = idx - h * D;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mm[w * kHeadsPerCta + h]);
        float L = 0.f, o = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float mw = mm[w * kHeadsPerCta + h];
            const float coef = mw == kNegInf ? 0.f : exp2_approx(mw - M);
            L += coef * ml[w * kHeadsPerCta + h];
            o += coef * mbuf[(w * kHeadsPerCta + h) * (D + 4) + d];
        }
        const float val = L > 0.f ? o / L : 0.f;
        const int64_t r = static_cast<int64_t>(seq) * a.num_q_heads + h0 + h;
        if (n_parts == 1) {
            store_out(a.out, r * D + d, val, a.out_dtype);
        } else {
            const int64_t pi = r * a.max_parts + part;
            a.part_o[pi * D + d] = val;
            if (d == 0) {
                a.part_ml[2 * pi] = M;
                a.part_ml[2 * pi + 1] = L;
            }
        }
    }
    if (n_parts > 1 && a.fused_merge)
        merge_group_if_last(a, seq, seq * gridDim.y + blockIdx.y, h0, nh, n_parts, threadIdx.x, blockDim.x,
                            [] { __syncthreads(); });
}

template <pa_dtype KV, int D>
pa_status launch(const DecodeArgs& a, cudaStream_t stream) {
    auto kernel = decode_simt_kernel<KV, D>;
    constexpr int smem = merge_floats<D>() * 4;
    static std::once_flag once;
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [&] { err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem); });
    if (err != cudaSuccess) return PA_ERR_CUDA;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    dim3 grid(a.max_parts, a.num_kv_heads * n_hg, a.batch);
    if (launch_pdl(kernel, grid, dim3(kWarps * 32), smem, stream, a) != cudaSuccess) return PA_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

template <pa_dtype KV>
pa_status launch_d(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch<KV, 64>(a, stream);
        case 128: return launch<KV, 128>(a, stream);
        case 256: return launch<KV, 256>(a, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace

pa_status launch_decode_simt(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.kv_dtype) {
        case PA_F32: return launch_d<PA_F32>(a, stream);
        case PA_F16: return launch_d<PA_F16>(a, stream);
        case PA_BF16: return launch_d<PA_BF16>(a, stream);
        case PA_FP8_E4M3: return launch_d<PA_FP8_E4M3>(a, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace pa
