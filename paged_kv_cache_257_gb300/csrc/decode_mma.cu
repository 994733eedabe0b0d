// Paged decode attention on the tensor cores (16-bit or FP8 cache, head_dim 128).
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 4 "The PagedAttention CUDA Kernel": the
// kernel reads the query, looks up the sequence's block table and fetches K
// and V from scattered physical blocks inside the attention loop; section 1
// gives softmax(Q K^T / sqrt(d_k)) V; section 2 Example 2: several query
// heads share one KV head (query head h reads KV head h / G).
//
// A work item is one (sequence, KV head, group of up to 8 of its query heads,
// partition of the context).  A CTA has four warps; chunk k of the item (16
// tokens) belongs to warp k % 4 and to ring stage k % NSTAGES, which only
// that warp uses:
//   * the warp walks the item's block table (32 ids per coalesced load) and
//     streams its chunks' K and V tiles into its stages with TMA loads
//     (128-byte swizzle, evict-first L2 hint; one 3-D box per 16-bit tile),
//     arming an mbarrier per stage, NSTAGES / 4 chunks ahead;
//   * for each chunk it forms S^T = K Q^T with mma.sync m16n8k16 (16 tokens
//     x 8 heads, heads on the N side so G = 8 needs no padding), runs the
//     online softmax in registers, turns P into the B operand with two
//     movmatrix transposes and accumulates O^T = V^T P^T;
//   * the warps' (max, sum, output) states are merged and written as the
//     final output or, for a split context, as a partition partial.
// The grid runs one CTA per item, 5 resident per SM.  FP8 tiles are widened
// to float16 in registers, with the K scale folded into the score scale and
// the V scale into the output.  A slid window ([start, ctx) of the row) masks
// the positions of its first chunk that precede the start.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "decode_epilogue.cuh"
#include "mma_chunk.cuh"
#include "window.cuh"

namespace pa {
namespace mma {

// ------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace {
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}
}  // namespace

// 2-D view of a pool: rows of head_dim elements, one row per (block, head,
// slot).  With `three_d`, a 3-D view (64 elements, rows, 2 column halves)
// whose box covers a whole 16-row tile.
bool make_pool_map(CUtensorMap* map, const void* pool, const DecodeArgs& a, int box_rows, bool three_d) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const int eb = static_cast<int>(pa_dtype_size(a.kv_dtype));
    CUtensorMapDataType t = a.kv_dtype == PA_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                            : a.kv_dtype == PA_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(kD),
                          static_cast<cuuint64_t>(a.num_blocks) * a.num_kv_heads * a.block_size};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(kD) * eb};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[3] = {1, 1, 1};
    if (three_d) {
        cuuint64_t dims3[3] = {static_cast<cuuint64_t>(128 / eb), dims[1], 2};
        cuuint64_t strides3[2] = {static_cast<cuuint64_t>(kD) * eb, 128};
        cuuint32_t box3[3] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows), 2};
        CUresult r = enc(map, t, 3, const_cast<void*>(pool), dims3, strides3, box3, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        return r == CUDA_SUCCESS;
    }
    CUresult r = enc(map, t, 2, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mma

namespace {

using namespace mma;

constexpr int kWarps = 4;         // warps per CTA, each loading and consuming its own stages
constexpr int kThreads = kWarps * 32;
constexpr int kDynTailChunks = 16;   // chunks at the end of an item shared out by a counter
constexpr int kMergeStride = kD + 4;  // floats per head row in merge buffers (bank spread)

template <pa_dtype KV, int BS, int NSTAGES>
struct Cfg : TileCfg<KV, BS> {
    static constexpr int kRingBytes = NSTAGES * TileCfg<KV, BS>::kStageBytes;
    // Chunk k goes to stage k % NSTAGES and to warp k % 4.  With
    // NSTAGES a multiple of 4 every stage always belongs to the same warp, so
    // that warp waits on the stage's phases strictly one after another and a
    // parity wait can never match a phase two fills old.  Any other depth
    // breaks that and must not be built.
    static_assert(NSTAGES % kWarps == 0, "each stage must belong to exactly one warp");
};

// Ring depth (16-token chunks in flight per CTA): a multiple of the
// warp count, small enough that 5 CTAs fit an SM.
#ifndef PA_DECODE_STAGES_16BIT
#define PA_DECODE_STAGES_16BIT 4
#endif
#ifndef PA_DECODE_STAGES_FP8
#define PA_DECODE_STAGES_FP8 8
#endif

// =====================================================================
// The kernel: one CTA per (partition, KV head group, sequence)
// =====================================================================

template <pa_dtype KV, int BS, int NSTAGES>
struct GridCfg : Cfg<KV, BS, NSTAGES> {
    using B = Cfg<KV, BS, NSTAGES>;
    // merge buffers: the warps' o rows, their (m, l) per head, the merged
    // (M, L) per head and a staging area for a partial's bulk store
    static constexpr int kMergeFloats =
        kWarps * (kHeadsPerCta * kMergeStride + 2 * kHeadsPerCta) + 2 * kHeadsPerCta + kHeadsPerCta * kD;
    static constexpr int kDataBytes = B::kRingBytes > kMergeFloats * 4 ? B::kRingBytes : kMergeFloats * 4;
    static constexpr int kSmemBytes = 1024 + kDataBytes + NSTAGES * 8;   // + one full barrier per stage
};

// Every warp streams its own stages: stage s belongs to warp s % 4, which
// issues its first NSTAGES / 4 chunks and, after consuming a chunk, has its
// lane 0 issue the chunk NSTAGES ahead into the stage just freed.  With no
// producer warp and no empty barriers a CTA is 4 warps, and the register
// budget at 5 CTAs per SM is 96 per thread (no spills).  A separate producer
// warp, tried first, left 72 registers (5 warps x 5 CTAs on 4 SM
// sub-partitions) and spilled: long-context FP8 ran 220 us against 182.
template <pa_dtype KV, int BS, int NSTAGES>
__global__ void __launch_bounds__(kThreads, PA_DECODE_MIN_CTAS)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeArgs a) {
    using C = GridCfg<KV, BS, NSTAGES>;
    constexpr bool kFp8 = KV == PA_FP8_E4M3;
    constexpr int S = NSTAGES / kWarps;   // stages per warp: warp w owns w, w + 4, ...

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);
    const uint32_t ring = smem_addr(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    const int kvh = blockIdx.y / n_hg, hg = blockIdx.y - kvh * n_hg;
    const int part = blockIdx.x;
    const int h0 = kvh * a.group + hg * kHeadsPerCta;
    const int nh = min(kHeadsPerCta, a.group - hg * kHeadsPerCta);
    const int32_t* bt_row = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;

    pdl_wait();      // inputs may come from the previous kernel in the stream
    pdl_trigger();
    WarpState<KV, C> cs;
    cs.init(lane);
    cs.reset();
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmap_k);
        prefetch_tmap(&tmap_v);
    }
    // The query, the context length and the partition's first 32 block ids
    // do not depend on one another: all are loaded before any is waited on.
    // The ids are a guess (blocks from part * P / block_size: right without
    // window starts when the partition share is P, and for partition 0),
    // used only once the real partition start confirms it.
    cs.template fetch_q<true>(static_cast<const uint16_t*>(a.q) + (static_cast<int64_t>(seq) * a.num_q_heads + h0) * kD,
                              nh);
    const bool spec = a.context_starts == nullptr;
    const int spec_j = part * (a.partition_size / BS) + lane;
    const int spec_ids = spec && spec_j < a.max_blocks ? __ldg(bt_row + spec_j) : 0;
    const SeqWindow sw = seq_window(a, seq, part == 0 && blockIdx.y == 0 && threadIdx.x == 0);
    const int n_parts = sw.n_parts;
    if (part >= n_parts) return;
    const int tok0 = sw.tok0(part);
    const int tok1 = sw.tok1(part);
    const int lead = sw.lead(part);   // positions of chunk 0 before the window
    const int n_chunks = tok1 > tok0 ? (tok1 - tok0 + kChunk - 1) / kChunk : 0;

    // the first chunk handed out by the counter below (a multiple of 4, past
    // the prologue's chunks)
    constexpr bool kClaims = S == 1;
    const int t_dyn = kClaims && a.balanced_tail ? max(NSTAGES, (n_chunks - kDynTailChunks) & ~(kWarps - 1))
                                                 : n_chunks + kWarps * S;   // past every chunk: no claims
    __shared__ int next_chunk;   // the next chunk no warp has taken yet
    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGES; ++i) mbar_init(smem_addr(full + i), 1);
        fence_mbar_init();
        next_chunk = t_dyn;
    }
    __syncthreads();
    const float sc = a.scale * 1.4426950408889634f * (kFp8 ? a.k_scale : 1.f);

    const uint64_t policy = l2_evict_first_policy();
    BlockWindow win;   // this warp's chunks, in increasing order
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
    // Chunk schedule.  Chunks below t_dyn go to the warps in a fixed
    // pattern: warp w takes w, w + 4, w + 8, ...  With one stage per warp
    // (16-bit caches) the last kDynTailChunks chunks are handed out in order
    // from a CTA-wide counter instead: a warp that has consumed a chunk takes
    // the next untaken one into the stage it just freed.  Warps whose copies
    // landed sooner take more of the tail, so the CTA's warps finish within
    // about one copy of one another; with the fixed pattern alone they ended
    // a median 2.7 us (up to 11 us) apart on the Llama-3-8B ragged batch,
    // which the tail counter makes 3% faster.  The counter stays out of the
    // rest of the loop: a claim per chunk (a shared-memory atomic and a
    // shuffle) made batches whose shared prefix is read from L2 4% slower.
    // FP8 warps (two copies in flight each) finish close together and keep
    // the fixed pattern to the end, as every warp does when the caller asked
    // for bit-reproducible results (a.balanced_tail == 0: which warp sums a
    // claimed chunk depends on timing, and with it the rounding of the
    // warp's probabilities).  Either way a warp's chunks come in
    // increasing order and its stages are used round robin: the k-th chunk
    // it consumes sits in stage warp + 4 (k % S) with phase (k / S) & 1.
    static_assert(!kClaims || S == 1, "claimed chunks are consumed in issue order only with one stage per warp");
    int issued = 0;   // this warp's chunks issued / consumed, in order
    for (int s = 0; s < S; ++s) {
        const int c = warp + kWarps * s;
        if (c < n_chunks) {
            issue(c, warp + kWarps * s);
            ++issued;
        }
    }
    // the query's widening waits for its loads: after the first copies are out
    cs.convert_q(a.q_dtype == PA_BF16);
    int k = 0;
    for (int c = warp; c < n_chunks; ++k) {
        const int st = warp + kWarps * (k % S);
        const bool landed = mbar_wait(smem_addr(full + st), (k / S) & 1);
        if (!__all_sync(0xffffffffu, landed)) {   // warp-uniform decision
            if (lane == 0) raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
            break;
        }
        int cn = c + kWarps * S;   // the chunk to bring into this stage next
        const bool claim = kClaims && cn >= t_dyn;   // warp-uniform
        if (claim && lane == 0) cn = atomicAdd(&next_chunk, 1);   // claimed now: its latency overlaps the math
        const uint32_t kb = ring + st * C::kStageBytes;
        cs.chunk(kb, kb + C::kTileBytes, c == 0 ? lead : 0, min(kChunk, tok1 - (tok0 + c * kChunk)), sc);
        __syncwarp();
        if (claim) cn = __shfl_sync(0xffffffffu, cn, 0);
        if (cn < n_chunks) {
            if (lane == 0) fence_proxy_async_smem();   // the reads above before the copy's writes
            issue(cn, st);
            ++issued;
        }
        // next to consume: with one stage per warp, the chunk just issued
        // (n_chunks or more: none); else the fixed pattern's next
        c = kClaims ? cn : c + kWarps;
    }
    // copies still in flight (only after a wait ran out): let them land
    // before the ring is reused
    if (lane == 0)
        for (int kk = k; kk < issued; ++kk)
            if (!mbar_wait(smem_addr(full + warp + kWarps * (kk % S)), (kk / S) & 1))
                raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
    cs.finish();

    __syncthreads();  // every stage consumed: the ring becomes the merge buffer

    float* mbuf = reinterpret_cast<float*>(smem);
    float* mm = mbuf + kWarps * kHeadsPerCta * kMergeStride;   // (warp, head): max, then the warp's weight
    float* ml = mm + kWarps * kHeadsPerCta;                    // (warp, head): row sum
    float* hml = ml + kWarps * kHeadsPerCta;                   // head: merged (M, L)
    float* stage = hml + 2 * kHeadsPerCta;                     // [head][kD]: a partial for its bulk store
    {
        float* w0 = mbuf + (warp * kHeadsPerCta + 2 * cs.q4) * kMergeStride;
        float* w1 = w0 + kMergeStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            w0[cs.d_lo(mt)] = cs.o[mt][0];
            w1[cs.d_lo(mt)] = cs.o[mt][1];
            w0[cs.d_hi(mt)] = cs.o[mt][2];
            w1[cs.d_hi(mt)] = cs.o[mt][3];
        }
        if (cs.g == 0) {
            mm[warp * kHeadsPerCta + 2 * cs.q4] = cs.m0;
            mm[warp * kHeadsPerCta + 2 * cs.q4 + 1] = cs.m1;
            ml[warp * kHeadsPerCta + 2 * cs.q4] = cs.l0;
            ml[warp * kHeadsPerCta + 2 * cs.q4 + 1] = cs.l1;
        }
    }
    __syncthreads();

    const float vs = kFp8 ? a.v_scale : 1.f;
    // Warp 0 weighs the warps' partial states once, lane = w * 8 + h:
    //     M_h = max_w m_wh,  L_h = sum_w 2^(m_wh - M_h) l_wh,
    //     weight_wh = 2^(m_wh - M_h) vs / L_h (0 for an empty head).
    // Every thread then only sums weighted o rows (with each thread redoing
    // the maxima, exponentials and sums, 128k-token FP8 contexts in
    // 512-token partitions ran 2.5% slower).
    static_assert(kWarps * kHeadsPerCta == 32, "one lane of warp 0 per (warp, head)");
    if (warp == 0) {
        const float m = mm[lane];
        float M = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, 16));
        const float coef = m == kNegInf ? 0.f : exp2_approx(m - M);
        float L = coef * ml[lane];
        L += __shfl_xor_sync(0xffffffffu, L, 8);
        L += __shfl_xor_sync(0xffffffffu, L, 16);
        mm[lane] = L > 0.f ? coef * vs / L : 0.f;   // each lane rewrites only its own entry
        if (lane < kHeadsPerCta) {
            hml[2 * lane] = M;
            hml[2 * lane + 1] = L;
        }
    }
    __syncthreads();

    // A split call's partials go out as one bulk copy per head when the merge
    // kernel reads them (its launch orders them), so that a CTA does not wait
    // on stores to a busy memory system; the fused merge's ticket needs its
    // partials visible first and keeps plain stores.
    const bool bulk = n_parts > 1 && !a.fused_merge;
    {
        const int d = threadIdx.x;   // 128 threads, one per element of head_dim
        // four heads at a time, unrolled (every warp wrote all kHeadsPerCta
        // heads; only the group's nh are stored).  Measured against a plain
        // loop over the nh heads: the same on most batches, 6% faster on a
        // batch whose shared prefix is read from L2.
        static_assert(kHeadsPerCta % 4 == 0, "heads are merged four at a time");
        for (int h4 = 0; h4 < nh; h4 += 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int h = h4 + j;
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w)
                    acc = fmaf(mm[w * kHeadsPerCta + h], mbuf[(w * kHeadsPerCta + h) * kMergeStride + d], acc);
                const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + h0 + h;
                if (h < nh) {
                    if (bulk)
                        stage[h * kD + d] = acc;
                    else
                        store_result(a, row, d, part, n_parts, acc, hml[2 * h], hml[2 * h + 1]);
                }
            }
        }
    }
    if (bulk) {
        const int64_t row0 = static_cast<int64_t>(seq) * a.num_q_heads + h0;
        if (threadIdx.x < nh) {   // (M, L) of one head: 8 bytes
            const int64_t pi = (row0 + threadIdx.x) * a.max_parts + part;
            reinterpret_cast<float2*>(a.part_ml)[pi] = make_float2(hml[2 * threadIdx.x], hml[2 * threadIdx.x + 1]);
        }
        fence_proxy_async_smem();   // the staged rows, written by every thread, before the copies read them
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int h = 0; h < nh; ++h)
                bulk_store(a.part_o + ((row0 + h) * a.max_parts + part) * kD, smem_addr(stage + h * kD), kD * 4);
            bulk_commit();
            bulk_wait_read();   // shared memory stays until the copies have read it
        }
    }
    if (n_parts > 1 && a.fused_merge) {
        merge_group_if_last(a, seq, seq * gridDim.y + blockIdx.y, h0, nh, n_parts, threadIdx.x, blockDim.x,
                            [] { __syncthreads(); });
    }
}

template <pa_dtype KV, int BS, int NSTAGES>
pa_status launch(const DecodeArgs& a, cudaStream_t stream) {
    CUtensorMap mk, mv;
    constexpr int box_rows = Cfg<KV, BS, NSTAGES>::kBoxRows;
    constexpr bool three_d = Cfg<KV, BS, NSTAGES>::k3D;
    if (!make_pool_map(&mk, a.k_cache, a, box_rows, three_d) || !make_pool_map(&mv, a.v_cache, a, box_rows, three_d))
        return PA_ERR_CUDA;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    using C = GridCfg<KV, BS, NSTAGES>;
    auto kernel = decode_mma_kernel<KV, BS, NSTAGES>;
    const int threads = kThreads;
    static std::once_flag once;   // once per instantiation
    static cudaError_t err = cudaSuccess;
    std::call_once(once, [&] { err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes); });
    if (err != cudaSuccess) return PA_ERR_CUDA;
    dim3 grid(a.max_parts, a.num_kv_heads * n_hg, a.batch);
    if (launch_pdl(kernel, grid, dim3(threads), C::kSmemBytes, stream, mk, mv, a) != cudaSuccess) return PA_ERR_CUDA;
    return PA_OK;
}

template <pa_dtype KV, int NSTAGES>
pa_status launch_bs(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.block_size) {
        case 8: return launch<KV, 8, NSTAGES>(a, stream);
        case 16: return launch<KV, 16, NSTAGES>(a, stream);
        case 32: return launch<KV, 32, NSTAGES>(a, stream);
    }
    return PA_ERR_UNSUPPORTED;
}

}  // namespace

bool mma_path_supported(const DecodeArgs& a) {
    if (a.head_dim != kD) return false;
    if (a.kv_dtype == PA_BF16) return a.q_dtype == PA_BF16;
    if (a.kv_dtype == PA_F16) return a.q_dtype == PA_F16;
    if (a.kv_dtype == PA_FP8_E4M3) return a.q_dtype == PA_BF16 || a.q_dtype == PA_F16;
    return false;
}

pa_status launch_decode_mma(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.kv_dtype) {
        case PA_BF16: return launch_bs<PA_BF16, PA_DECODE_STAGES_16BIT>(a, stream);
        case PA_F16: return launch_bs<PA_F16, PA_DECODE_STAGES_16BIT>(a, stream);
        case PA_FP8_E4M3: return launch_bs<PA_FP8_E4M3, PA_DECODE_STAGES_FP8>(a, stream);
        default: return PA_ERR_UNSUPPORTED;
    }
}

}  // namespace pa
