// Paged decode attention on the tensor cores (16-bit or FP8 cache, head_dim 128).
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 4 "The PagedAttention CUDA Kernel": the
// kernel reads the query, looks up the sequence's block table and fetches K
// and V from scattered physical blocks inside the attention loop; section 1
// gives softmax(Q K^T / sqrt(d_k)) V; section 2 Example 2: several query
// heads share one KV head (query head h reads KV head h / G).
//
// One CTA serves one (partition of the context, KV head, sequence) and up to
// eight query heads of that KV head's group.  Four consumer warps and one
// producer warp:
//   * the producer walks the block table (32 ids per coalesced load) and
//     streams each 16-token chunk's K and V tiles into a ring of shared
//     memory stages with 2-D TMA loads (128-byte swizzle, evict-first L2
//     hint), signalling an mbarrier per stage;
//   * consumer warp w takes chunks w, w+4, ...; for each it forms
//     S^T = K Q^T with mma.sync m16n8k16 (16 tokens x 8 heads, the heads on
//     the N side so G = 8 needs no padding), runs the online softmax in
//     registers, turns P into the B operand with two movmatrix transposes
//     and accumulates O^T = V^T P^T (8 tiles of 16 rows of head_dim);
//   * the warps' (max, sum, output) states are merged in shared memory and
//     written either as the final output or, for a split context, as a
//     partition partial that a second kernel merges.
// FP8 tiles are widened to float16 in registers (exact), with the K scale
// folded into the score scale and the V scale into the output.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "decode.h"
#include "decode_epilogue.cuh"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kChunk = 16;        // tokens per mma row tile
constexpr int kConsumers = 4;     // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kMergeStride = kD + 4;  // floats per head row in the merge buffer (bank spread)
constexpr float kNegInf = -__builtin_huge_valf();

template <pa_dtype KV, int BS, int NSTAGES>
struct Cfg {
    static constexpr int kElemBytes = Elem<KV>::bytes;
    static constexpr int kHalves = kD * kElemBytes / 128;    // 128-byte column halves of a row
    static constexpr int kRegionBytes = kChunk * 128;        // 16 rows x 128 B, one swizzle unit
    static constexpr int kTileBytes = kHalves * kRegionBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;       // K tile then V tile
    static constexpr int kBoxRows = BS < kChunk ? BS : kChunk;
    static constexpr int kBoxBytes = kBoxRows * 128;
    static constexpr int kRingBytes = NSTAGES * kStageBytes;
    static constexpr int kMergeFloats = kConsumers * (kHeadsPerCta * kMergeStride + 2 * kHeadsPerCta);
    static constexpr int kDataBytes = kRingBytes > kMergeFloats * 4 ? kRingBytes : kMergeFloats * 4;
    static constexpr int kSmemBytes = 1024 + kDataBytes + 2 * NSTAGES * 8 + 16;
    static_assert(kD * kElemBytes % 128 == 0, "rows must be whole 128-byte swizzle spans");
    // Chunk c goes to stage c % NSTAGES and to consumer warp c % 4.  With
    // NSTAGES a multiple of 4 every stage always belongs to the same warp, so
    // that warp waits on the stage's phases strictly one after another and a
    // parity wait can never match a phase two fills old.  Any other depth
    // breaks that and must not be built.
    static_assert(NSTAGES % kConsumers == 0, "each stage must belong to exactly one consumer warp");
};

// Ring depth (16-token chunks in flight per CTA): a multiple of the consumer
// warp count, small enough that 4 CTAs fit an SM.
#ifndef PA_DECODE_STAGES_16BIT
#define PA_DECODE_STAGES_16BIT 4
#endif
#ifndef PA_DECODE_STAGES_FP8
#define PA_DECODE_STAGES_FP8 8
#endif

// Largest growth (log2 units) of a chunk's score maximum over the running
// reference before the accumulators are rescaled.
constexpr float kLazyRescale = 8.f;

// O^T[128 d][8 heads] += V^T P^T for one 16-token chunk held in stage `vb`.
// 16-bit caches: ldmatrix.trans gives the A fragments directly.  FP8: each
// ldmatrix.trans register holds (token 2q: d, d+1 | token 2q+1: d, d+1); a
// byte permute regroups it into token pairs at a fixed d before widening, so
// m-tile rows interleave d (row i <-> d = 16 mt + 2 i, row i + 8 <-> + 1).
template <pa_dtype KV, typename C, bool MASK>
__device__ __forceinline__ void pv_chunk(float (&o)[8][4], uint32_t vb, uint32_t v_row, int v_sel, int sw,
                                         uint32_t pb0, uint32_t pb1, uint32_t vm01, uint32_t vm23) {
    if constexpr (KV != PA_FP8_E4M3) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t ar[4];
            ldsm_x4_t(vb + (mt >> 2) * C::kRegionBytes + v_row + ((((mt & 3) * 2 + v_sel) ^ sw) << 4), ar[0], ar[1],
                      ar[2], ar[3]);
            if constexpr (MASK) {
                ar[0] &= vm01; ar[1] &= vm01; ar[2] &= vm23; ar[3] &= vm23;
            }
            mma_16816<KV == PA_BF16>(o[mt], ar, pb0, pb1);
        }
    } else {
#pragma unroll
        for (int c2 = 0; c2 < 4; ++c2) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(vb + v_row + (((2 * c2 + v_sel) ^ sw) << 4), r0, r1, r2, r3);
            uint32_t ar[4], br[4];
            e4m3x4_to_f16x2x2(byte_perm(r0, 0, 0x3120), ar[0], ar[1]);   // tokens 0..7, d / d+1
            e4m3x4_to_f16x2x2(byte_perm(r2, 0, 0x3120), ar[2], ar[3]);   // tokens 8..15
            e4m3x4_to_f16x2x2(byte_perm(r1, 0, 0x3120), br[0], br[1]);
            e4m3x4_to_f16x2x2(byte_perm(r3, 0, 0x3120), br[2], br[3]);
            if constexpr (MASK) {
                ar[0] &= vm01; ar[1] &= vm01; ar[2] &= vm23; ar[3] &= vm23;
                br[0] &= vm01; br[1] &= vm01; br[2] &= vm23; br[3] &= vm23;
            }
            mma_16816<false>(o[2 * c2], ar, pb0, pb1);
            mma_16816<false>(o[2 * c2 + 1], br, pb0, pb1);
        }
    }
}

template <pa_dtype KV, int BS, int NSTAGES>
__global__ void __launch_bounds__(kThreads, 4)
decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                  const DecodeArgs a) {
    using C = Cfg<KV, BS, NSTAGES>;
    constexpr bool kFp8 = KV == PA_FP8_E4M3;
    constexpr bool kBf16 = KV == PA_BF16;  // mma operand type: bf16, else f16

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kDataBytes);
    uint64_t* empty = full + NSTAGES;
    int* abort_flag = reinterpret_cast<int*>(empty + NSTAGES);
    const uint32_t ring = smem_addr(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seq = blockIdx.z;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    const int kvh = blockIdx.y / n_hg, hg = blockIdx.y - kvh * n_hg;
    const int part = blockIdx.x;

    pdl_wait();      // inputs may come from the previous kernel in the stream
    pdl_trigger();
    int ctx = __ldg(a.context_lens + seq);
    const int cap = a.max_blocks * BS;
    if (ctx < 0 || ctx > cap) {
        if (part == 0 && blockIdx.y == 0 && threadIdx.x == 0) raise_flag(a.status, PA_DEVFLAG_CONTEXT_RANGE);
        ctx = ctx < 0 ? 0 : cap;
    }
    const int n_parts = ctx > 0 ? (ctx + a.partition_size - 1) / a.partition_size : 1;
    if (part >= n_parts) return;
    const int tok0 = part * a.partition_size;
    const int tok1 = min(ctx, tok0 + a.partition_size);
    const int n_chunks = tok1 > tok0 ? (tok1 - tok0 + kChunk - 1) / kChunk : 0;
    const int h0 = kvh * a.group + hg * kHeadsPerCta;
    const int nh = min(kHeadsPerCta, a.group - hg * kHeadsPerCta);

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTAGES; ++i) {
            mbar_init(smem_addr(full + i), 1);
            mbar_init(smem_addr(empty + i), 1);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // consumer state (registers), kept across the block-wide barriers below
    float o[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;

    if (warp == kConsumers) {
        // ------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tmap(&tmap_k);
            prefetch_tmap(&tmap_v);
        }
        const uint64_t policy = l2_evict_first_policy();
        const int32_t* bt = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks;
        const int j_first = tok0 / BS;
        const int j_end = n_chunks > 0 ? (tok1 - 1) / BS + 1 : j_first;  // exclusive
        int id_base = -32, my_id = 0;
        int issued = 0;
        for (int c = 0; c < n_chunks; ++c) {
            const int st = c % NSTAGES;
            if (c >= NSTAGES) {
                int ok = 1;
                if (lane == 0) ok = mbar_wait(smem_addr(empty + st), ((c / NSTAGES) - 1) & 1);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) {
                        atomicExch(abort_flag, 1);
                        raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
                    }
                    break;
                }
                if (*reinterpret_cast<volatile int*>(abort_flag)) break;
            }
            const int t0 = tok0 + c * kChunk;
            const int rel = t0 / BS - j_first;   // window-relative index of the chunk's first block
            if (rel >= id_base + 32) {
                id_base = rel & ~31;
                const int j = j_first + id_base + lane;
                my_id = j < j_end ? __ldg(bt + j) : 0;
            }
            int pb_a = __shfl_sync(0xffffffffu, my_id, rel - id_base);
            int pb_b = 0;
            if constexpr (BS < kChunk) pb_b = __shfl_sync(0xffffffffu, my_id, (rel + 1 - id_base) & 31);
            if (lane == 0) {
                const bool two = BS < kChunk && t0 + BS < tok1;   // second block holds valid tokens
                if (pb_a < 0 || pb_a >= a.num_blocks) {
                    raise_flag(a.status, PA_DEVFLAG_BLOCK_RANGE);
                    pb_a = a.num_blocks;   // rows past the tensor: TMA fills zeros
                }
                if (two && (pb_b < 0 || pb_b >= a.num_blocks)) {
                    raise_flag(a.status, PA_DEVFLAG_BLOCK_RANGE);
                    pb_b = a.num_blocks;
                }
                const int boxes = (two ? 2 : 1) * C::kHalves * 2;
                const uint32_t fb = smem_addr(full + st);
                mbar_arrive_expect_tx(fb, boxes * C::kBoxBytes);
                const uint32_t kdst = ring + st * C::kStageBytes;
                const int ya = (pb_a * a.num_kv_heads + kvh) * BS + (t0 % BS);
                const int yb = (pb_b * a.num_kv_heads + kvh) * BS;
#pragma unroll
                for (int hf = 0; hf < C::kHalves; ++hf) {
                    const int x = hf * (128 / C::kElemBytes);
                    const uint32_t kd = kdst + hf * C::kRegionBytes;
                    const uint32_t vd = kd + C::kTileBytes;
                    tma_load_2d(kd, &tmap_k, fb, x, ya, policy);
                    tma_load_2d(vd, &tmap_v, fb, x, ya, policy);
                    if (two) {
                        tma_load_2d(kd + C::kBoxBytes, &tmap_k, fb, x, yb, policy);
                        tma_load_2d(vd + C::kBoxBytes, &tmap_v, fb, x, yb, policy);
                    }
                }
            }
            ++issued;
            __syncwarp();
        }
        // every copy this CTA issued has landed before shared memory is reused
        if (lane == 0) {
            for (int st = 0; st < NSTAGES && st < issued; ++st) {
                const int fills = (issued - st + NSTAGES - 1) / NSTAGES;
                if (!mbar_wait(smem_addr(full + st), (fills - 1) & 1)) raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
            }
        }
    } else {
        // ------------------------------------------------------ consumers
        const int g = lane >> 2;   // fragment group: row (token) / column (head) index
        const int q4 = lane & 3;   // thread in group
        const float sc = a.scale * 1.4426950408889634f * (kFp8 ? a.k_scale : 1.f);

        // Q as the B operand of S^T = K Q^T: column n = head g, 16 rows of d per k-step
        uint32_t qf[8][2];
        {
            const bool hv = g < nh;
            const int64_t qrow = (static_cast<int64_t>(seq) * a.num_q_heads + h0 + (hv ? g : 0)) * kD;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                if constexpr (!kFp8) {
                    const uint32_t* qp = static_cast<const uint32_t*>(a.q);
                    qf[kk][0] = hv ? __ldg(qp + (qrow + 16 * kk + 2 * q4) / 2) : 0u;
                    qf[kk][1] = hv ? __ldg(qp + (qrow + 16 * kk + 8 + 2 * q4) / 2) : 0u;
                } else {
                    // FP8 tiles arrive as 4 consecutive codes per k pair (see the K loop):
                    // k rows (2q, 2q+1) <-> d = 16kk + 4q + {0,1}, (2q+8, 2q+9) <-> d + {2,3}
                    const int64_t e = qrow + 16 * kk + 4 * q4;
                    const uint2 raw = hv ? __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(a.q) + e))
                                         : make_uint2(0u, 0u);
                    if (a.q_dtype == PA_BF16) {   // bf16 -> float (exact) -> f16
                        qf[kk][0] = pack2<false>(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u));
                        qf[kk][1] = pack2<false>(__uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
                    } else {
                        qf[kk][0] = raw.x;
                        qf[kk][1] = raw.y;
                    }
                }
            }
        }

        // per-lane parts of the swizzled shared-memory addresses (row & 7 == lane & 7)
        const int sw = lane & 7;
        const uint32_t k_row = ((lane & 7) + 8 * ((lane >> 3) & 1)) * 128;   // ldmatrix rows of K
        const uint32_t v_row = ((lane & 7) + 8 * (lane >> 4)) * 128;         // ldmatrix rows of V
        const int k_sel = lane >> 4;          // K: second 16-byte column of the pair
        const int v_sel = (lane >> 3) & 1;    // V: second 16-byte column of the pair

        for (int c = warp; c < n_chunks; c += kConsumers) {
            const int st = c % NSTAGES;
            const bool landed = mbar_wait(smem_addr(full + st), (c / NSTAGES) & 1);
            if (!__all_sync(0xffffffffu, landed)) {   // warp-uniform decision
                if (lane == 0) {
                    atomicExch(abort_flag, 1);
                    raise_flag(a.status, PA_DEVFLAG_TIMEOUT);
                }
                break;
            }
            const uint32_t kb = ring + st * C::kStageBytes;
            const uint32_t vb = kb + C::kTileBytes;

            // ---- S^T[16 tokens][8 heads] = K Q^T, as two independent accumulation chains
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (!kFp8) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    uint32_t ar[4];
                    const uint32_t addr = kb + (kk >> 2) * C::kRegionBytes + k_row +
                                          ((((kk & 3) * 2 + k_sel) ^ sw) << 4);
                    ldsm_x4(addr, ar[0], ar[1], ar[2], ar[3]);
                    mma_16816<kBf16>((kk & 1) ? sb : sa, ar, qf[kk][0], qf[kk][1]);
                }
            } else {
#pragma unroll
                for (int c2 = 0; c2 < 4; ++c2) {
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(kb + k_row + (((2 * c2 + k_sel) ^ sw) << 4), r0, r1, r2, r3);
                    uint32_t ar[4], br[4];
                    e4m3x4_to_f16x2x2(r0, ar[0], ar[2]);   // row g:   d+{0,1} | d+{2,3}
                    e4m3x4_to_f16x2x2(r1, ar[1], ar[3]);   // row g+8
                    mma_16816<false>(sa, ar, qf[2 * c2][0], qf[2 * c2][1]);
                    e4m3x4_to_f16x2x2(r2, br[0], br[2]);
                    e4m3x4_to_f16x2x2(r3, br[1], br[3]);
                    mma_16816<false>(sb, br, qf[2 * c2 + 1][0], qf[2 * c2 + 1][1]);
                }
            }

            // ---- online softmax over this chunk (log2 domain)
            const int valid = tok1 - (tok0 + c * kChunk);   // >= 1; < 16 only in the last chunk
            float x0 = (sa[0] + sb[0]) * sc, x1 = (sa[1] + sb[1]) * sc;
            float x2 = (sa[2] + sb[2]) * sc, x3 = (sa[3] + sb[3]) * sc;
            if (valid < kChunk) {
                if (g >= valid) x0 = x1 = kNegInf;
                if (g + 8 >= valid) x2 = x3 = kNegInf;
            }
            float cm0 = fmaxf(x0, x2), cm1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                cm0 = fmaxf(cm0, __shfl_xor_sync(0xffffffffu, cm0, off));
                cm1 = fmaxf(cm1, __shfl_xor_sync(0xffffffffu, cm1, off));
            }
            // The reference maximum moves only when a score exceeds it by more than
            // 2^kLazyRescale; until then p <= 2^kLazyRescale and (m, l, o) stay
            // consistent, so the rescale of o is skipped on most chunks.
            if (__any_sync(0xffffffffu, cm0 > m0 + kLazyRescale || cm1 > m1 + kLazyRescale)) {
                const float mn0 = fmaxf(m0, cm0), mn1 = fmaxf(m1, cm1);
                const float al0 = exp2_approx(m0 - mn0), al1 = exp2_approx(m1 - mn1);   // 0 on the first chunk
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    o[i][0] *= al0; o[i][1] *= al1;
                    o[i][2] *= al0; o[i][3] *= al1;
                }
                m0 = mn0;
                m1 = mn1;
            }
            const float p0 = exp2_approx(x0 - m0), p2 = exp2_approx(x2 - m0);
            const float p1 = exp2_approx(x1 - m1), p3 = exp2_approx(x3 - m1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            // P^T as the B operand: (token, head) pairs transposed to (head, token)
            const uint32_t pb0 = movmatrix_t(pack2<kBf16>(p0, p1));   // tokens 0..7
            const uint32_t pb1 = movmatrix_t(pack2<kBf16>(p2, p3));   // tokens 8..15

            // ---- O^T[128 d][8 heads] += V^T P^T; in the last chunk the rows past
            // the context hold stale stage data, so their V is zeroed first
            if (valid < kChunk) {
                const uint32_t vm01 = (2 * q4 < valid ? 0x0000ffffu : 0u) | (2 * q4 + 1 < valid ? 0xffff0000u : 0u);
                const uint32_t vm23 = (2 * q4 + 8 < valid ? 0x0000ffffu : 0u) | (2 * q4 + 9 < valid ? 0xffff0000u : 0u);
                pv_chunk<KV, C, true>(o, vb, v_row, v_sel, sw, pb0, pb1, vm01, vm23);
            } else {
                pv_chunk<KV, C, false>(o, vb, v_row, v_sel, sw, pb0, pb1, 0u, 0u);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(empty + st));
        }
        // row sums were kept per lane; add over the 8 lanes sharing a head pair
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
    }

    __syncthreads();  // every stage consumed (or drained): the ring becomes the merge buffer

    float* mbuf = reinterpret_cast<float*>(smem);
    float* mm = mbuf + kConsumers * kHeadsPerCta * kMergeStride;
    float* ml = mm + kConsumers * kHeadsPerCta;
    if (warp < kConsumers) {
        const int g = lane >> 2, q4 = lane & 3;
        float* w0 = mbuf + (warp * kHeadsPerCta + 2 * q4) * kMergeStride;
        float* w1 = w0 + kMergeStride;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            const int d_lo = kFp8 ? 16 * mt + 2 * g : 16 * mt + g;
            const int d_hi = kFp8 ? d_lo + 1 : d_lo + 8;
            w0[d_lo] = o[mt][0];
            w1[d_lo] = o[mt][1];
            w0[d_hi] = o[mt][2];
            w1[d_hi] = o[mt][3];
        }
        if (g == 0) {
            mm[warp * kHeadsPerCta + 2 * q4] = m0;
            mm[warp * kHeadsPerCta + 2 * q4 + 1] = m1;
            ml[warp * kHeadsPerCta + 2 * q4] = l0;
            ml[warp * kHeadsPerCta + 2 * q4 + 1] = l1;
        }
    }
    __syncthreads();

    if (threadIdx.x < kD) {
        const int d = threadIdx.x;
        const float vs = kFp8 ? a.v_scale : 1.f;
        for (int h = 0; h < nh; ++h) {
            float M = kNegInf;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, mm[w * kHeadsPerCta + h]);
            float L = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < kConsumers; ++w) {
                const float mw = mm[w * kHeadsPerCta + h];
                const float coef = mw == kNegInf ? 0.f : exp2_approx(mw - M);
                L += coef * ml[w * kHeadsPerCta + h];
                acc += coef * mbuf[(w * kHeadsPerCta + h) * kMergeStride + d];
            }
            const float val = L > 0.f ? acc * vs / L : 0.f;
            const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + h0 + h;
            if (n_parts == 1) {
                store_out(a.out, row * kD + d, val, a.out_dtype);
            } else {
                const int64_t pi = row * a.max_parts + part;
                a.part_o[pi * kD + d] = val;
                if (d == 0) {
                    a.part_ml[2 * pi] = M;
                    a.part_ml[2 * pi + 1] = L;
                }
            }
        }
    }
    if (n_parts > 1 && a.fused_merge) merge_if_last(a, seq, h0, nh, n_parts);
}

// ------------------------------------------------------------ host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// 2-D view of a pool: rows of head_dim elements, one row per (block, head, slot).
bool make_pool_map(CUtensorMap* map, const void* pool, const DecodeArgs& a, int box_rows) {
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
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, t, 2, const_cast<void*>(pool), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <pa_dtype KV, int BS, int NSTAGES>
pa_status launch(const DecodeArgs& a, cudaStream_t stream) {
    using C = Cfg<KV, BS, NSTAGES>;
    auto kernel = decode_mma_kernel<KV, BS, NSTAGES>;
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [&] {
        attr_err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return PA_ERR_CUDA;
    CUtensorMap mk, mv;
    if (!make_pool_map(&mk, a.k_cache, a, C::kBoxRows) || !make_pool_map(&mv, a.v_cache, a, C::kBoxRows))
        return PA_ERR_CUDA;
    const int n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    dim3 grid(a.max_parts, a.num_kv_heads * n_hg, a.batch);
    if (launch_pdl(kernel, grid, dim3(kThreads), C::kSmemBytes, stream, mk, mv, a) != cudaSuccess) return PA_ERR_CUDA;
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
