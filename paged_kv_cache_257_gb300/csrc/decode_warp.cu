// Paged decode attention with one warp per work item (16-bit or FP8 cache,
// head_dim 128), for problems with many long work items.
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 4 "The PagedAttention CUDA Kernel": the
// kernel reads the query, looks up the sequence's block table and fetches K
// and V from scattered physical blocks inside the attention loop; section 1
// gives softmax(Q K^T / sqrt(d_k)) V; section 2 Example 2: query head h reads
// KV head h / G.
//
// A work item is one (sequence, KV head, group of up to 8 of its query heads,
// partition of the context), as in the CTA-per-item kernel, but here one
// warp is the whole CTA: it walks the item's block table, keeps S chunks of
// 16 tokens in flight in its own stages (TMA loads, 128-byte swizzle,
// evict-first L2 hint), and runs every chunk through the same per-chunk step
// (mma.sync S^T = K Q^T, online softmax, O^T += V^T P^T).  Its softmax state
// is the item's result, so there is no cross-warp merge, no CTA barrier and
// no merge buffer: an item ends with the warp's rows normalised in
// registers, staged in its ring and written out, while up to 20 such warps
// per SM keep their copies in flight (20 with FP8 caches; with 16-bit
// caches the two 8 KB stages per warp let shared memory hold 11).  When items are long and many (a
// 128k-token FP8 context in 512-token partitions gives 8192 of 32 chunks), a
// CTA of four warps spends a third of its life filling its pipeline and
// merging its warps; independent warps remove the merge and let every other
// warp on the SM stream through one warp's start-up.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "decode_epilogue.cuh"
#include "mma_chunk.cuh"
#include "window.cuh"

namespace pa {
namespace {

using namespace mma;

// Chunks in flight per warp.
#ifndef PA_WARP_STAGES_FP8
#define PA_WARP_STAGES_FP8 2
#endif
#ifndef PA_WARP_STAGES_16BIT
#define PA_WARP_STAGES_16BIT 2
#endif

constexpr int kOutStride = kD + 4;   // floats per staged result row (bank spread)

template <pa_dtype KV, int BS, int S>
struct WarpCfg : TileCfg<KV, BS> {
    using T = TileCfg<KV, BS>;
    static constexpr int kRingBytes = S * T::kStageBytes;
    static constexpr int kResultBytes = kHeadsPerCta * kOutStride * 4;   // [head][kOutStride] floats
    static constexpr int kDataBytes = kRingBytes > kResultBytes ? kRingBytes : kResultBytes;
    static constexpr int kSmemBytes = 1024 + kDataBytes + S * 8;         // + one full barrier per stage
};

// One warp per CTA and per item; registers sized for PA_DECODE_WARP_MIN_CTAS
// resident per SM (shared memory allows that many with FP8 caches, 11 with
// 16-bit ones).
template <pa_dtype KV, int BS, int S>
__global__ void __launch_bounds__(32, PA_DECODE_WARP_MIN_CTAS)
decode_warp_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                   const DecodeArgs a) {
    using C = WarpCfg<KV, BS, S>;
    constexpr bool kFp8 = KV == PA_FP8_E4M3;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);
    const uint32_t ring = smem_addr(smem);

    const int lane = threadIdx.x;
    const int seq = blockIdx.z;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    const int kvh = blockIdx.y / n_hg, hg = blockIdx.y - kvh * n_hg;
    const int part = blockIdx.x;
    const int h0 = kvh * a.group + hg * kHeadsPerCta;
    const int nh = min(kHeadsPerCta, a.group - hg * kHeadsPerCta);
    const int32_t* bt_row = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;

    // The barriers need no inputs: set them up before anything is loaded.
    if (lane == 0) {
        for (int i = 0; i < S; ++i) mbar_init(smem_addr(full + i), 1);
        fence_mbar_init();
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    pdl_wait();      // inputs may come from the previous kernel in the stream
    pdl_trigger();
    WarpState<KV, C> cs;
    cs.init(lane);
    cs.reset();
    // The query, the context length and the partition's first 32 block ids
    // are loaded before any is waited on; the ids are a guess (blocks from
    // part * P / block_size), used only once the real partition start
    // confirms it.
    cs.template fetch_q<true>(static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(seq) * a.num_q_heads + h0) * kD,
                              nh);
    const bool spec = a.context_starts == nullptr;
    const int spec_j = part * (a.partition_size / BS) + lane;
    const int spec_ids = spec && spec_j < a.max_blocks ? __ldg(bt_row + spec_j) : 0;
    const SeqWindow sw = seq_window(a, seq, part == 0 && blockIdx.y == 0 && lane == 0);
    const int n_parts = sw.n_parts;
    if (part >= n_parts) return;
    const int tok0 = sw.tok0(part);
    const int tok1 = sw.tok1(part);
    const int lead = sw.lead(part);   // positions of chunk 0 before the window
    const int n_chunks = tok1 > tok0 ? (tok1 - tok0 + kChunk - 1) / kChunk : 0;

    __syncwarp();
    const float sc = a.scale * 1.4426950408889634f * (kFp8 ? a.k_scale : 1.f);

    const uint64_t policy = l2_evict_first_policy();
    BlockWindow win;   // the item's chunks, in increasing order
    if (spec && tok0 == part * a.partition_size)
        win.start_loaded(bt_row, tok0, tok1, BS, spec_ids);
    else
        win.start(bt_row, tok0, tok1, BS);
    auto issue = [&](int c, int st) {   // the whole warp: the block ids come by shuffle
        const int t0 = tok0 + c * kChunk;
        int pb_a, pb_b;
        win.get(t0, BS, lane, pb_a, pb_b);
        // an 8-token block wholly before a slid window may have been
        // released: its rows (masked anyway) come from the chunk's second block
        if (BS < kChunk && c == 0 && lead >= BS) pb_a = pb_b;
        issue_tiles<C, BS>(a, &tmap_k, &tmap_v, full, ring, st, lane, kvh, t0, tok1, pb_a, pb_b, policy);
    };
    // Chunk c lives in stage c % S with phase (c / S) & 1; after consuming
    // it the warp issues chunk c + S into the same stage.
    int issued = 0;
    for (int c = 0; c < S && c < n_chunks; ++c) {
        issue(c, c);
        ++issued;
    }
    // the query's widening waits for its loads: after the first copies are out
    cs.convert_q(a.q_dtype == PA_BF16);
    int c = 0;
    for (; c < n_chunks; ++c) {
        const int st = c % S;
        const bool landed = mbar_wait(smem_addr(full + st), (c / S) & 1);
        if (!__all_sync(0xffffffffu, landed)) {   // warp-uniform decision
            if (lane == 0) raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
            break;
        }
        const uint32_t kb = ring + st * C::kStageBytes;
        cs.chunk(kb, kb + C::kTileBytes, c == 0 ? lead : 0, min(kChunk, tok1 - (tok0 + c * kChunk)), sc);
        __syncwarp();
        if (c + S < n_chunks) {
            if (lane == 0) fence_proxy_async_smem();   // the reads above before the copy's writes
            issue(c + S, st);
            ++issued;
        }
    }
    // copies still in flight (only after a wait ran out): let them land
    // before the ring holds the result
    if (lane == 0)
        for (int kk = c; kk < issued; ++kk)
            if (!mbar_wait(smem_addr(full + kk % S), (kk / S) & 1)) raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
    cs.finish();
    __syncwarp();

    // The item's rows o / l (x the V scale), staged as [head][kOutStride]
    // floats so that each head leaves as one coalesced 512-byte row.
    const float vs = kFp8 ? a.v_scale : 1.f;
    const float w0 = cs.l0 > 0.f ? vs / cs.l0 : 0.f;
    const float w1 = cs.l1 > 0.f ? vs / cs.l1 : 0.f;
    float* res = reinterpret_cast<float*>(smem);
    {
        float* r0 = res + (2 * cs.q4) * kOutStride;
        float* r1 = r0 + kOutStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            r0[cs.d_lo(mt)] = cs.o[mt][0] * w0;
            r1[cs.d_lo(mt)] = cs.o[mt][1] * w1;
            r0[cs.d_hi(mt)] = cs.o[mt][2] * w0;
            r1[cs.d_hi(mt)] = cs.o[mt][3] * w1;
        }
    }
    __syncwarp();
    const int64_t row0 = static_cast<int64_t>(seq) * a.num_q_heads + h0;
    if (n_parts == 1) {
        for (int h = 0; h < nh; ++h) {
            const float4 v = *reinterpret_cast<const float4*>(res + h * kOutStride + 4 * lane);
            const int64_t i = (row0 + h) * kD + 4 * lane;
            store_out(a.out, i, v.x, a.out_dtype);
            store_out(a.out, i + 1, v.y, a.out_dtype);
            store_out(a.out, i + 2, v.z, a.out_dtype);
            store_out(a.out, i + 3, v.w, a.out_dtype);
        }
        return;
    }
    for (int h = 0; h < nh; ++h) {
        const float4 v = *reinterpret_cast<const float4*>(res + h * kOutStride + 4 * lane);
        *reinterpret_cast<float4*>(a.part_o + ((row0 + h) * a.max_parts + part) * kD + 4 * lane) = v;
    }
    if (cs.g == 0) {   // lanes 0..3 hold the (max, sum) of heads 2q, 2q + 1
        const int ha = 2 * cs.q4, hb = ha + 1;
        if (ha < nh)
            reinterpret_cast<float2*>(a.part_ml)[(row0 + ha) * a.max_parts + part] = make_float2(cs.m0, cs.l0);
        if (hb < nh)
            reinterpret_cast<float2*>(a.part_ml)[(row0 + hb) * a.max_parts + part] = make_float2(cs.m1, cs.l1);
    }
    if (a.fused_merge)
        merge_group_if_last(a, seq, seq * gridDim.y + blockIdx.y, h0, nh, n_parts, lane, 32, [] { __syncwarp(); });
}

template <pa_dtype KV, int BS, int S>
pa_status launch(const DecodeArgs& a, cudaStream_t stream) {
    using C = WarpCfg<KV, BS, S>;
    CUtensorMap mk, mv;
    if (!make_pool_map(&mk, a.k_cache, a, C::kBoxRows, C::k3D) || !make_pool_map(&mv, a.v_cache, a, C::kBoxRows, C::k3D))
        return PA_ERR_CUDA;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    auto kernel = decode_warp_kernel<KV, BS, S>;
    static std::once_flag once;   // once per instantiation
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [&] { err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes); });
    if (err != cudaSuccess) return PA_ERR_CUDA;
    dim3 grid(a.max_parts, a.num_kv_heads * n_hg, a.batch);
    if (launch_pdl(kernel, grid, dim3(32), C::kSmemBytes, stream, mk, mv, a) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

template <pa_dtype KV, int S>
pa_status launch_bs(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.block_size) {
        case 8: return launch<KV, 8, S>(a, stream);
        case 16: return launch<KV, 16, S>(a, stream);
        case 32: return launch<KV, 32, S>(a, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace

pa_status launch_decode_warp(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.kv_dtype) {
        case PA_BF16: return launch_bs<PA_BF16, PA_WARP_STAGES_16BIT>(a, stream);
        case PA_F16: return launch_bs<PA_F16, PA_WARP_STAGES_16BIT>(a, stream);
        case PA_FP8_E4M3: return launch_bs<PA_FP8_E4M3, PA_WARP_STAGES_FP8>(a, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace pa
