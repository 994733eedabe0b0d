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
    // The output is nh x D floats, handled as float4 slices (D is a multiple
    // of 4), two per thread and pass, the partitions four at a time.  The
    // first pass's partial outputs are loaded before the (max, sum) pairs
    // are read, so that both loads take one round trip between them.
    const int slices = nh * D / 4;
    auto load = [&](int i, int p0, float4 (&v)[4]) {
        const int h = (4 * i) / D, d = 4 * i - h * D;
        const float* po = a.part_o + ((row0 + h) * a.max_parts + p0) * D + d;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            v[j] = i < slices && p0 + j < n_parts ? __ldcg(reinterpret_cast<const float4*>(po + j * D))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    float4 v0[4], v1[4];
    load(tid, 0, v0);
    load(tid + nthreads, 0, v1);
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
    for (int i = tid; i < slices; i += 2 * nthreads) {
        const int i1 = i + nthreads;
        const int ha = (4 * i) / D, hb = min((4 * i1) / D, nh - 1);   // hb: clamped for a missing second slice
        float4 acc0 = make_float4(0.f, 0.f, 0.f, 0.f), acc1 = acc0;
        for (int p0 = 0; p0 < n_parts; p0 += 4) {
            if (i != tid || p0 != 0) {   // the first pass was loaded above
                load(i, p0, v0);
                load(i1, p0, v1);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float wa = p0 + j < n_parts ? s_w[ha][p0 + j] : 0.f;
                const float wb = p0 + j < n_parts && i1 < slices ? s_w[hb][p0 + j] : 0.f;
                acc0.x = fmaf(wa, v0[j].x, acc0.x);
                acc0.y = fmaf(wa, v0[j].y, acc0.y);
                acc0.z = fmaf(wa, v0[j].z, acc0.z);
                acc0.w = fmaf(wa, v0[j].w, acc0.w);
                acc1.x = fmaf(wb, v1[j].x, acc1.x);
                acc1.y = fmaf(wb, v1[j].y, acc1.y);
                acc1.z = fmaf(wb, v1[j].z, acc1.z);
                acc1.w = fmaf(wb, v1[j].w, acc1.w);
            }
        }
        const int64_t oa = row0 * D + 4 * i;
        store_out(a.out, oa, acc0.x, a.out_dtype);
        store_out(a.out, oa + 1, acc0.y, a.out_dtype);
        store_out(a.out, oa + 2, acc0.z, a.out_dtype);
        store_out(a.out, oa + 3, acc0.w, a.out_dtype);
        if (i1 < slices) {
            const int64_t ob = row0 * D + 4 * i1;
            store_out(a.out, ob, acc1.x, a.out_dtype);
            store_out(a.out, ob + 1, acc1.y, a.out_dtype);
            store_out(a.out, ob + 2, acc1.z, a.out_dtype);
            store_out(a.out, ob + 3, acc1.w, a.out_dtype);
        }
    }
    if (tid == 0) a.tickets[grp] = 0;
}

}  // namespace pa
