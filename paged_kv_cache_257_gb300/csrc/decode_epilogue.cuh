// Fused split-context merge, shared by the decode kernels.
//
// When a sequence's context spans several partitions, each partition's CTA
// writes its partial (max m, sum l, normalised output o) for its query heads,
// then takes a ticket for its (sequence, KV head, head group).  The CTA that
// draws the last ticket merges the group's partials
//     M = max_p m_p,  w_p = l_p 2^(m_p - M),  out = sum_p w_p o_p / sum_p w_p
// and resets the ticket to zero, so the ticket array is zero again after
// every call.  No CTA ever waits for another: the ticket is a plain atomic
// counter (the threadfence-reduction pattern).  Used when the number of
// partitions is small; large counts go to the separate merge kernel.
#pragma once

#include "common.cuh"
#include "decode.h"

namespace pa {

__device__ __forceinline__ void merge_if_last(const DecodeArgs& a, int seq, int h0, int nh, int n_parts) {
    __shared__ int s_last;
    const int grp = seq * gridDim.y + blockIdx.y;   // (sequence, KV head, head group)
    __threadfence();                                // this CTA's partials before its ticket
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(a.tickets + grp, 1) == n_parts - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();                                // every partial of the group is visible
    const float neg_inf = -__builtin_huge_valf();
    const int D = a.head_dim;
    for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
        const int h = idx / D, d = idx - h * D;
        const int64_t row = static_cast<int64_t>(seq) * a.num_q_heads + h0 + h;
        const float* ml = a.part_ml + row * a.max_parts * 2;
        const float* po = a.part_o + row * a.max_parts * D + d;
        float M = neg_inf;
        for (int p = 0; p < n_parts; ++p) M = fmaxf(M, __ldcg(ml + 2 * p));
        float L = 0.f, acc = 0.f;
        for (int p = 0; p < n_parts; ++p) {
            const float mp = __ldcg(ml + 2 * p);
            const float w = mp == neg_inf ? 0.f : __ldcg(ml + 2 * p + 1) * exp2_approx(mp - M);
            L += w;
            acc = fmaf(w, __ldcg(po + static_cast<int64_t>(p) * D), acc);
        }
        store_out(a.out, row * D + d, L > 0.f ? acc / L : 0.f, a.out_dtype);
    }
    if (threadIdx.x == 0) a.tickets[grp] = 0;
}

}  // namespace pa
