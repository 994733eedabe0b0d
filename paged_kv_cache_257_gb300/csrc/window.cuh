// The positions of a sequence that decode attends, and their partitions.
//
// A sequence attends the positions [start, ctx) of its block-table row:
// start is 0 unless the caller slid the window (vaibhawkumar.in "Why LLMs run
// out of VRAM: KV cache fragmentation and the PagedAttention fix", "A minimal
// PyTorch sketch", truncate: whole leading pages are released and the rest of
// the drop is an offset into the first kept page).  The window, counted from
// base = start rounded down to a multiple of 16, splits into
// n = ceil((ctx - base) / P) partitions of equal length S (the share rounded
// up to the partition unit, max(16, block size); S <= P and the last
// partition is never empty): partition p covers [base + p*S, min(ctx, base +
// (p+1)*S)).  Equal shares keep the work items of a ragged batch alike in
// size; a length that is a multiple of P gives partitions of exactly P.
// Every 16-token chunk starts on a chunk boundary of the row (a whole
// 16-token block, half a 32-token block, or two 8-token blocks) and only the
// first chunk of partition 0 holds positions before start.  An empty window
// (start == ctx) is one partition of no tokens: output 0.
#pragma once

#include "common.cuh"
#include "decode.h"

namespace pa {

struct SeqWindow {
    int ctx, start, base, n_parts, share;   // share: tokens per partition (S)
    __device__ __forceinline__ int tok0(int part) const { return base + part * share; }
    __device__ __forceinline__ int tok1(int part) const {
        const int t0 = tok0(part);
        return ctx > start ? min(ctx, t0 + share) : t0;
    }
    // positions of partition `part`'s first chunk that precede the window
    __device__ __forceinline__ int lead(int part) const { return part == 0 ? start - base : 0; }
};

// Context length and start of sequence `seq`, clamped to the row (a value
// out of range raises PA_DEVFLAG_CONTEXT_RANGE when `report`).
__device__ __forceinline__ SeqWindow seq_window(const DecodeArgs& a, int seq, bool report) {
    int ctx = __ldg(a.context_lens + seq);
    const int cap = a.max_blocks * a.block_size;
    if (ctx < 0 || ctx > cap) {
        if (report) raise_flag(a.status, PA_DEVFLAG_CONTEXT_RANGE);
        ctx = ctx < 0 ? 0 : cap;
    }
    int start = a.context_starts != nullptr ? __ldg(a.context_starts + seq) : 0;
    if (start < 0 || start > ctx) {
        if (report) raise_flag(a.status, PA_DEVFLAG_CONTEXT_RANGE);
        start = start < 0 ? 0 : ctx;
    }
    SeqWindow w;
    w.ctx = ctx;
    w.start = start;
    w.base = start & ~15;
    const int len = ctx - w.base;
    const int unit = a.block_size > 16 ? a.block_size : 16;
    w.n_parts = ctx > start ? (len + a.partition_size - 1) / a.partition_size : 1;
    w.share = ctx > start ? ((len + w.n_parts - 1) / w.n_parts + unit - 1) / unit * unit : a.partition_size;
    return w;
}

}  // namespace pa
