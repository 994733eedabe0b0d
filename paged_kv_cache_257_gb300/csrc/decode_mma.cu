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
#include "window.cuh"

namespace pa {
namespace {

constexpr int kD = 128;
constexpr int kChunk = 16;        // tokens per mma row tile
constexpr int kWarps = 4;         // warps per CTA, each loading and consuming its own stages
constexpr int kThreads = kWarps * 32;
constexpr int kDynTailChunks = 16;   // chunks at the end of an item shared out by a counter
constexpr int kMergeStride = kD + 4;  // floats per head row in merge buffers (bank spread)
constexpr float kNegInf = -__builtin_huge_valf();

// 1: 16-bit tiles with 16-row boxes move as one 3-D TMA box (128-byte
// column halves as the outermost box dimension, so shared memory still holds
// [half][row][128 B]); 0: one 2-D box per half.
#ifndef PA_TMA_3D
#define PA_TMA_3D 1
#endif

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
    static constexpr bool k3D = PA_TMA_3D && kHalves == 2 && kBoxRows == kChunk;   // one box per tile
    static_assert(kD * kElemBytes % 128 == 0, "rows must be whole 128-byte swizzle spans");
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

// FP8 tiles are widened to float16 for the tensor cores with
// cvt.rn.f16x2.e4m3x2 on pairs of codes (exact values).  Moving the E4M3 bit
// fields into float16 positions instead (values x 2^-8, folded into the
// scales; 7 integer operations per four codes, no byte permute) ran 273 us
// against 242 us on the long-context FP8 workload.

// K operand: the four codes a thread holds of one row (d+0..3) as the A
// fragment's (k 2q, 2q+1) and (k 2q+8, 2q+9) registers; the query is loaded
// in the same d order.
__device__ __forceinline__ void fp8_k_pairs(uint32_t x, uint32_t& k01, uint32_t& k89) {
    e4m3x4_to_f16x2x2(x, k01, k89);           // d+{0,1} | d+{2,3}
}

// V operand: an ldmatrix.trans register (token 2q: d, d+1 | token 2q+1: d, d+1)
// as the token pairs at d and at d+1.
__device__ __forceinline__ void fp8_v_pairs(uint32_t x, uint32_t& at_d, uint32_t& at_d1) {
    e4m3x4_to_f16x2x2(__byte_perm(x, 0, 0x3120), at_d, at_d1);
}

// Largest growth (log2 units) of a chunk's score maximum over the running
// reference before the accumulators are rescaled.
constexpr float kLazyRescale = 8.f;

// O^T[128 d][8 heads] += V^T P^T for one 16-token chunk held in stage `vb`.
// 16-bit caches: ldmatrix.trans gives the A fragments directly.  FP8: each
// ldmatrix.trans register holds (token 2q: d, d+1 | token 2q+1: d, d+1),
// regrouped into token pairs at a fixed d while widening, so m-tile rows
// interleave d (row i <-> d = 16 mt + 2 i, row i + 8 <-> + 1).
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
            fp8_v_pairs(r0, ar[0], ar[1]);   // tokens 0..7 at d | d+1
            fp8_v_pairs(r2, ar[2], ar[3]);   // tokens 8..15
            fp8_v_pairs(r1, br[0], br[1]);
            fp8_v_pairs(r3, br[2], br[3]);
            if constexpr (MASK) {
                ar[0] &= vm01; ar[1] &= vm01; ar[2] &= vm23; ar[3] &= vm23;
                br[0] &= vm01; br[1] &= vm01; br[2] &= vm23; br[3] &= vm23;
            }
            mma_16816<false>(o[2 * c2], ar, pb0, pb1);
            mma_16816<false>(o[2 * c2 + 1], br, pb0, pb1);
        }
    }
}

// One warp's online-softmax state for up to 8 query heads (lane
// holds heads 2q, 2q+1) and its per-chunk step.
template <pa_dtype KV, typename C>
struct WarpState {
    static constexpr bool kFp8 = KV == PA_FP8_E4M3;
    static constexpr bool kBf16 = KV == PA_BF16;   // mma operand type: bf16, else f16
    float o[8][4];
    float m0, m1, l0, l1;
    uint32_t qf[8][2];
    int g, q4, sw, k_sel, v_sel;
    uint32_t k_row, v_row;

    __device__ __forceinline__ void init(int lane) {
        g = lane >> 2;     // fragment group: row (token) / column (head) index
        q4 = lane & 3;     // thread in group
        sw = lane & 7;     // swizzle phase (row & 7 == lane & 7 for every ldmatrix below)
        k_row = ((lane & 7) + 8 * ((lane >> 3) & 1)) * 128;   // ldmatrix rows of K
        v_row = ((lane & 7) + 8 * (lane >> 4)) * 128;         // ldmatrix rows of V
        k_sel = lane >> 4;                                    // K: second 16-byte column of the pair
        v_sel = (lane >> 3) & 1;                              // V: second 16-byte column of the pair
    }

    __device__ __forceinline__ void reset() {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        m0 = m1 = kNegInf;
        l0 = l1 = 0.f;
    }

    // Q as the B operand of S^T = K Q^T: column n = head g, 16 rows of d per
    // k-step.  `rows` points at the first head's row (nh rows of kD 16-bit
    // elements); GLOBAL selects read-only global loads over generic ones.
    // load_q = fetch_q (the loads alone, so a caller can overlap them with
    // other waits) then convert_q (FP8 caches: the query widened to f16 in the
    // K operand's d order).
    template <bool GLOBAL>
    __device__ __forceinline__ void fetch_q(const uint16_t* rows, int nh) {
        const bool hv = g < nh;
        const uint16_t* row = rows + (hv ? g : 0) * kD;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            if constexpr (!kFp8) {
                const uint32_t* p0 = reinterpret_cast<const uint32_t*>(row + 16 * kk + 2 * q4);
                const uint32_t* p1 = reinterpret_cast<const uint32_t*>(row + 16 * kk + 8 + 2 * q4);
                qf[kk][0] = hv ? (GLOBAL ? __ldg(p0) : *p0) : 0u;
                qf[kk][1] = hv ? (GLOBAL ? __ldg(p1) : *p1) : 0u;
            } else {
                // FP8 tiles give each thread 4 consecutive codes per row and k-step
                // (d = 16kk + 4q + 0..3): the query's d = 16kk + 4q + 0..3 raw
                const uint2* p = reinterpret_cast<const uint2*>(row + 16 * kk + 4 * q4);
                const uint2 raw = hv ? (GLOBAL ? __ldg(p) : *p) : make_uint2(0u, 0u);
                qf[kk][0] = raw.x;
                qf[kk][1] = raw.y;
            }
        }
    }
    __device__ __forceinline__ void convert_q(bool q_bf16) {
        if constexpr (kFp8) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t h01 = qf[kk][0], h23 = qf[kk][1];
                if (q_bf16) {   // bf16 -> float (exact) -> f16
                    h01 = pack2<false>(__uint_as_float(h01 << 16), __uint_as_float(h01 & 0xffff0000u));
                    h23 = pack2<false>(__uint_as_float(h23 << 16), __uint_as_float(h23 & 0xffff0000u));
                }
                qf[kk][0] = h01;   // d+0, d+1: ordered like fp8_k_pairs
                qf[kk][1] = h23;   // d+2, d+3
            }
        }
    }
    template <bool GLOBAL>
    __device__ __forceinline__ void load_q(const uint16_t* rows, int nh, bool q_bf16) {
        fetch_q<GLOBAL>(rows, nh);
        convert_q(q_bf16);
    }

    // One 16-token chunk in stage (kb: K tile, vb: V tile); its tokens lo..hi-1
    // are attended (0 <= lo < hi <= 16: lo > 0 only for the chunk holding a slid
    // window's start, hi < 16 only at the context's end); `sc` = softmax scale
    // x log2(e) (x K scale).
    __device__ __forceinline__ void chunk(uint32_t kb, uint32_t vb, int lo, int hi, float sc) {
        // ---- S^T[16 tokens][8 heads] = K Q^T, as two independent accumulation chains
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (!kFp8) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t ar[4];
                const uint32_t addr = kb + (kk >> 2) * C::kRegionBytes + k_row + ((((kk & 3) * 2 + k_sel) ^ sw) << 4);
                ldsm_x4(addr, ar[0], ar[1], ar[2], ar[3]);
                mma_16816<kBf16>((kk & 1) ? sb : sa, ar, qf[kk][0], qf[kk][1]);
            }
        } else {
#pragma unroll
            for (int c2 = 0; c2 < 4; ++c2) {
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kb + k_row + (((2 * c2 + k_sel) ^ sw) << 4), r0, r1, r2, r3);
                uint32_t ar[4], br[4];
                fp8_k_pairs(r0, ar[0], ar[2]);   // row g
                fp8_k_pairs(r1, ar[1], ar[3]);   // row g+8
                mma_16816<false>(sa, ar, qf[2 * c2][0], qf[2 * c2][1]);
                fp8_k_pairs(r2, br[0], br[2]);
                fp8_k_pairs(r3, br[1], br[3]);
                mma_16816<false>(sb, br, qf[2 * c2 + 1][0], qf[2 * c2 + 1][1]);
            }
        }

        // ---- online softmax over this chunk (log2 domain)
        float x0 = (sa[0] + sb[0]) * sc, x1 = (sa[1] + sb[1]) * sc;
        float x2 = (sa[2] + sb[2]) * sc, x3 = (sa[3] + sb[3]) * sc;
        const bool partial = lo > 0 || hi < kChunk;
        if (partial) {
            if (g < lo || g >= hi) x0 = x1 = kNegInf;
            if (g + 8 < lo || g + 8 >= hi) x2 = x3 = kNegInf;
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

        // ---- O^T[128 d][8 heads] += V^T P^T; rows outside lo..hi-1 hold stale
        // stage data (or another block's), so their V is zeroed first
        if (partial) {
            auto in = [&](int t) { return t >= lo && t < hi; };
            const uint32_t vm01 = (in(2 * q4) ? 0x0000ffffu : 0u) | (in(2 * q4 + 1) ? 0xffff0000u : 0u);
            const uint32_t vm23 = (in(2 * q4 + 8) ? 0x0000ffffu : 0u) | (in(2 * q4 + 9) ? 0xffff0000u : 0u);
            pv_chunk<KV, C, true>(o, vb, v_row, v_sel, sw, pb0, pb1, vm01, vm23);
        } else {
            pv_chunk<KV, C, false>(o, vb, v_row, v_sel, sw, pb0, pb1, 0u, 0u);
        }
    }

    // Row sums were kept per lane; add over the 8 lanes sharing a head pair.
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
    }

    // d of this lane's accumulator o[mt][0/1] (lo) and o[mt][2/3] (hi)
    __device__ __forceinline__ int d_lo(int mt) const { return kFp8 ? 16 * mt + 2 * g : 16 * mt + g; }
    __device__ __forceinline__ int d_hi(int mt) const { return kFp8 ? 16 * mt + 2 * g + 1 : 16 * mt + g + 8; }
};

// Test builds only (never the library's default build): arm each stage for
// this many bytes more than its copies bring, so that no stage ever
// completes and every wait runs into its time limit.  This is how the tests
// check that a stalled copy ends in PA_DEVFLAG_TIMEOUT, not a hang.
#ifndef PA_TEST_EXTRA_TX
#define PA_TEST_EXTRA_TX 0
#endif

// Lane 0 arms stage st's full barrier with the chunk's byte count and
// issues its K and V boxes (the stage must be free).  `pb_a` / `pb_b` are the
// physical blocks of the chunk's first / second block (the second only for
// 8-token blocks).
template <typename C, int BS>
__device__ __forceinline__ void issue_tiles(const DecodeArgs& a, const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                            uint64_t* full, uint32_t ring, int st, int lane, int kvh, int t0,
                                            int tok1, int pb_a, int pb_b, uint64_t policy) {
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
        mbar_arrive_expect_tx(fb, boxes * C::kBoxBytes + PA_TEST_EXTRA_TX);
        const uint32_t kdst = ring + st * C::kStageBytes;
        const int ya = (pb_a * a.num_kv_heads + kvh) * BS + (t0 % BS);
        const int yb = (pb_b * a.num_kv_heads + kvh) * BS;
        if constexpr (C::k3D) {
            tma_load_3d(kdst, tmap_k, fb, 0, ya, 0, policy);
            tma_load_3d(kdst + C::kTileBytes, tmap_v, fb, 0, ya, 0, policy);
        } else {
#pragma unroll
            for (int hf = 0; hf < C::kHalves; ++hf) {
                const int x = hf * (128 / C::kElemBytes);
                const uint32_t kd = kdst + hf * C::kRegionBytes;
                const uint32_t vd = kd + C::kTileBytes;
                tma_load_2d(kd, tmap_k, fb, x, ya, policy);
                tma_load_2d(vd, tmap_v, fb, x, ya, policy);
                if (two) {
                    tma_load_2d(kd + C::kBoxBytes, tmap_k, fb, x, yb, policy);
                    tma_load_2d(vd + C::kBoxBytes, tmap_v, fb, x, yb, policy);
                }
            }
        }
    }
}

// Block ids of an item's chunks, 32 at a time from one coalesced load.
struct BlockWindow {
    const int32_t* bt;
    int j_first, j_end, base, my_id;
    __device__ __forceinline__ void start(const int32_t* table, int tok0, int tok1, int bs) {
        bt = table;
        j_first = tok0 / bs;
        j_end = tok1 > tok0 ? (tok1 - 1) / bs + 1 : j_first;
        base = -32;
        my_id = 0;
    }
    // the same, with the first 32 ids (blocks j_first + lane) already loaded
    __device__ __forceinline__ void start_loaded(const int32_t* table, int tok0, int tok1, int bs, int ids) {
        start(table, tok0, tok1, bs);
        base = 0;
        my_id = ids;
    }
    // physical blocks of the chunk starting at token t0 (second: t0 + 8, for 8-token blocks)
    __device__ __forceinline__ void get(int t0, int bs, int lane, int& pb_a, int& pb_b) {
        const int rel = t0 / bs - j_first;
        if (rel >= base + 32) {
            base = rel & ~31;
            const int j = j_first + base + lane;
            my_id = j < j_end ? __ldg(bt + j) : 0;
        }
        pb_a = __shfl_sync(0xffffffffu, my_id, rel - base);
        pb_b = __shfl_sync(0xffffffffu, my_id, (rel + 1 - base) & 31);
    }
};

// Write one merged value: the final output, or this partition's partial.
__device__ __forceinline__ void store_result(const DecodeArgs& a, int64_t row, int d, int part, int n_parts,
                                             float val, float M, float L) {
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
    cs.convert_q(a.q_dtype == PA_BF16);

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
