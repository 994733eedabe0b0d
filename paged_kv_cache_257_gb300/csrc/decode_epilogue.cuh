// Fused split-context merge, shared by the decode kernels.
//
// When a sequence's context spans several partitions, each partition's CTA
// writes its partial (max m, sum l, normalised output o) for its query heads,
// then takes a ticket for its (sequence, KV head, head group).  The CTA that
// draws the last ticket merges the group's partials
//     M = max_p m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// and resets the ticket to zero, so the ticket array is zero again after
// every call.  No CTA ever waits for another: the ticket is a plain atomic
// counter (the threadfence-reduction pattern).  Used when a sequence has at
// most kFusedMergeMaxParts partitions; larger counts go to the merge kernel.
#pragma once

#include "common.cuh"
#include "decode.h"

namespace pa {

// Run by `nthreads` threads (ids `tid`) that synchronise through `bar`;
// `grp` indexes the (sequence, KV head, head group) ticket.
template <typename Bar>
__device__ __forceinline__ void merge_group_if_last(const DecodeArgs& a, int seq, int grp, int h0, int nh,
                                                    int n_parts, int tid, int nthreads, Bar bar) {
    __shared__ int s_last;
    __shared__ float s_m[kHeadsPerCta][kFusedMergeMaxParts];
    __shared__ float s_w[kHeadsPerCta][kFusedMergeMaxParts];
    bar();                                          // every partial of this CTA is written
    if (tid == 0) {
        __threadfence();                            // ... and visible before the ticket
        const bool last = atomicAdd(a.tickets + grp, 1) == n_parts - 1;
        if (last) __threadfence();                  // the other CTAs' partials are visible
        s_last = last;
    }
    bar();
    if (!s_last) return;
    const float neg_inf = -__builtin_huge_valf();
    const int D = a.head_dim;
    const int64_t row0 = static_cast<int64_t>(seq) * a.num_q_heads + h0;
    // every (head, partition) pair's max and sum, one per thread
    for (int i = tid; i < nh * n_parts; i += nthreads) {
        const int h = i / n_parts, p = i - h * n_parts;
        const float* ml = a.part_ml + ((row0 + h) * a.max_parts + p) * 2;
        s_m[h][p] = __ldcg(ml);
        s_w[h][p] = __ldcg(ml + 1);
    }
    bar();
    if (tid < nh) {                                 // per head: weights normalised by their sum
        const int h = tid;
        float M = neg_inf;
        for (int p = 0; p < n_parts; ++p) M = fmaxf(M, s_m[h][p]);
        float L = 0.f;
        for (int p = 0; p < n_parts; ++p) {
            const float w = s_m[h][p] == neg_inf ? 0.f : s_w[h][p] * exp2_approx(s_m[h][p] - M);
            s_w[h][p] = w;
            L += w;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int p = 0; p < n_parts; ++p) s_w[h][p] *= inv;
    }
    bar();
    for (int idx = tid; idx < nh * D; idx += nthreads) {
        const int h = idx / D, d = idx - h * D;
        const float* po = a.part_o + (row0 + h) * a.max_parts * D + d;
        float v[kFusedMergeMaxParts];
#pragma unroll
        for (int p = 0; p < kFusedMergeMaxParts; ++p) v[p] = p < n_parts ? __ldcg(po + p * D) : 0.f;
        float acc = 0.f;
#pragma unroll
        for (int p = 0; p < kFusedMergeMaxParts; ++p) acc = p < n_parts ? fmaf(s_w[h][p], v[p], acc) : acc;
        store_out(a.out, (row0 + h) * D + d, acc, a.out_dtype);
    }
    if (tid == 0) a.tickets[grp] = 0;
}

}  // namespace pa
