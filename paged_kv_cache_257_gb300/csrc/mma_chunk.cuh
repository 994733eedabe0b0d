// The per-chunk machinery of the tensor-core decode kernels: tile geometry
// of a 16-token chunk in shared memory, its TMA loads, the block-table
// window that names its physical blocks, and one warp's online-softmax
// state with its step over a chunk (S^T = K Q^T, softmax, O^T += V^T P^T on
// mma.sync m16n8k16).  Shared by the CTA-per-item kernel (four warps split
// an item's chunks) and the warp-per-item kernel (one warp streams a whole
// item).
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 4 "The PagedAttention CUDA Kernel": read
// the query, look up the block table, fetch K and V from scattered blocks;
// section 1: softmax(Q K^T / sqrt(d_k)) V; section 2 Example 2: query head h
// reads KV head h / G.
#pragma once

#include "common.cuh"
#include "decode.h"

namespace pa {
namespace mma {


constexpr int kD = 128;
constexpr int kChunk = 16;        // tokens per mma row tile
constexpr float kNegInf = -__builtin_huge_valf();

// 1: 16-bit tiles with 16-row boxes move as one 3-D TMA box (128-byte
// column halves as the outermost box dimension, so shared memory still holds
// [half][row][128 B]); 0: one 2-D box per half.
#ifndef PA_TMA_3D
#define PA_TMA_3D 1
#endif

template <pa_dtype KV, int BS>
struct TileCfg {
    static constexpr int kElemBytes = Elem<KV>::bytes;
    static constexpr int kHalves = kD * kElemBytes / 128;    // 128-byte column halves of a row
    static constexpr int kRegionBytes = kChunk * 128;        // 16 rows x 128 B, one swizzle unit
    static constexpr int kTileBytes = kHalves * kRegionBytes;
    static constexpr int kStageBytes = 2 * kTileBytes;       // K tile then V tile
    static constexpr int kBoxRows = BS < kChunk ? BS : kChunk;
    static constexpr int kBoxBytes = kBoxRows * 128;
    static constexpr bool k3D = PA_TMA_3D && kHalves == 2 && kBoxRows == kChunk;   // one box per tile
    static_assert(kD * kElemBytes % 128 == 0, "rows must be whole 128-byte swizzle spans");
};

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

// Tensor map of a pool for the chunk loads: 2-D rows of head_dim elements,
// one row per (block, head, slot), 128-byte boxes of `box_rows` rows; with
// `three_d`, a 3-D view (64 elements, rows, 2 column halves) whose box
// covers a whole 16-row tile of a 16-bit pool.
bool make_pool_map(CUtensorMap* map, const void* pool, const DecodeArgs& a, int box_rows, bool three_d);

}  // namespace mma
}  // namespace pa
