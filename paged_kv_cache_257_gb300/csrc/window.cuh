// The positions of a sequence that decode attends, and their partitions.
//
// A sequence attends the positions [start, ctx) of its block-table row:
// start is 0 unless the caller slid the window (vaibhawkumar.in "Why LLMs run
// out of VRAM: KV cache fragmentation and the PagedAttention fix", "A minimal
// PyTorch sketch", truncate: whole leading pages are released and the rest of
// the drop is an offset into the first kept page).  Partition p covers
// [base + p*P, min(ctx, base + (p+1)*P)) with base = start rounded down to a
// multiple of 16, so every 16-token chunk starts on a chunk boundary of the
// row (a whole 16-token block, half a 32-token block, or two 8-token blocks)
// and only the first chunk of partition 0 holds positions before start.  An
// empty window (start == ctx) is one partition of no tokens: output 0.
#pragma once

#include "common.cuh"
#include "decode.h"

namespace pa {

struct SeqWindow {
    int ctx, start, base, n_parts;
    __device__ __forceinline__ int tok0(int part, int partition_size) const { return base + part * partition_size; }
    __device__ __forceinline__ int tok1(int part, int partition_size) const {
        const int t0 = tok0(part, partition_size);
        return ctx > start ? min(ctx, t0 + partition_size) : t0;
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
    w.n_parts = ctx > start ? (ctx - w.base + a.partition_size - 1) / a.partition_size : 1;
    return w;
}

}  // namespace pa
