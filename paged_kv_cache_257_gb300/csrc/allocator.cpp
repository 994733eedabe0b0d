// Host block allocator: LIFO free pool, reference counts, copy-on-write.
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 4 "How the Architecture Works": one pool
// of physical blocks allocated up front, a new block taken when a sequence's
// last block fills; section 5 "Zero-Copy Forking": forked sequences share
// blocks under a reference count, and a branch's first write into a shared
// block gets a private copy.  hyperinfer.ai "KV cache & paged attention deep
// dive", "What 16-token blocks buy you": evicting a sequence frees its blocks.
// vaibhawkumar.in "Why LLMs run out of VRAM: KV cache fragmentation and the
// PagedAttention fix", "PagedAttention: the idea" and "A minimal PyTorch
// sketch" (truncate): sliding the window releases the oldest whole pages and
// keeps the rest of the drop as an offset into the first kept page.
#include <algorithm>
#include <cstdint>
#include <new>
#include <unordered_map>
#include <vector>

#include "pagedattn.h"

struct pa_allocator {
    int32_t num_blocks;
    std::vector<int32_t> free_stack;  // top = back()
    std::vector<int32_t> ref;
};

namespace {

// SplitMix64 (Steele, Lea & Flood, 2014): state += golden gamma, then the
// two xor-shift-multiply rounds of its output function.
struct SplitMix64 {
    uint64_t state;
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ULL;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
        return z ^ (z >> 31);
    }
};

bool valid_id(const pa_allocator* a, int32_t b) { return b >= 0 && b < a->num_blocks; }

}  // namespace

extern "C" {

pa_status pa_alloc_create(int32_t num_blocks, uint64_t seed, pa_allocator** out) {
    if (out == nullptr) return PA_ERR_INVALID;
    *out = nullptr;
    if (num_blocks <= 0) return PA_ERR_INVALID;
    pa_allocator* a = new (std::nothrow) pa_allocator;
    if (a == nullptr) return PA_ERR_OOM;
    a->num_blocks = num_blocks;
    std::vector<int32_t> order(static_cast<size_t>(num_blocks));
    for (int32_t i = 0; i < num_blocks; ++i) order[i] = i;
    if (seed != 0) {  // Durstenfeld's Fisher-Yates, i from n-1 down to 1
        SplitMix64 rng{seed};
        for (int32_t i = num_blocks - 1; i > 0; --i) {
            uint64_t j = rng.next() % static_cast<uint64_t>(i + 1);
            int32_t t = order[i];
            order[i] = order[j];
            order[j] = t;
        }
    }
    // hand-out order is order[0], order[1], ...: the stack top is order[0]
    a->free_stack.assign(order.rbegin(), order.rend());
    a->ref.assign(static_cast<size_t>(num_blocks), 0);
    *out = a;
    return PA_OK;
}

void pa_alloc_destroy(pa_allocator* a) { delete a; }

int32_t pa_alloc_num_blocks(const pa_allocator* a) { return a ? a->num_blocks : 0; }

int32_t pa_alloc_free_count(const pa_allocator* a) {
    return a ? static_cast<int32_t>(a->free_stack.size()) : 0;
}

int32_t pa_alloc_refcount(const pa_allocator* a, int32_t block) {
    if (a == nullptr || !valid_id(a, block)) return -1;
    return a->ref[block];
}

pa_status pa_alloc_block(pa_allocator* a, int32_t* block_out) {
    if (a == nullptr || block_out == nullptr) return PA_ERR_INVALID;
    if (a->free_stack.empty()) return PA_ERR_OOM;
    int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->ref[b] = 1;
    *block_out = b;
    return PA_OK;
}

pa_status pa_alloc_incref(pa_allocator* a, int32_t block) {
    if (a == nullptr) return PA_ERR_INVALID;
    if (!valid_id(a, block)) return PA_ERR_RANGE;
    if (a->ref[block] == 0) return PA_ERR_INVALID;
    a->ref[block] += 1;
    return PA_OK;
}

pa_status pa_alloc_decref(pa_allocator* a, int32_t block) {
    if (a == nullptr) return PA_ERR_INVALID;
    if (!valid_id(a, block)) return PA_ERR_RANGE;
    if (a->ref[block] == 0) return PA_ERR_INVALID;
    if (--a->ref[block] == 0) a->free_stack.push_back(block);
    return PA_OK;
}

pa_status pa_alloc_cow(pa_allocator* a, int32_t block, int32_t* new_block_out, int32_t* copied) {
    if (a == nullptr || new_block_out == nullptr || copied == nullptr) return PA_ERR_INVALID;
    if (!valid_id(a, block)) return PA_ERR_RANGE;
    if (a->ref[block] == 0) return PA_ERR_INVALID;
    if (a->ref[block] == 1) {
        *new_block_out = block;
        *copied = 0;
        return PA_OK;
    }
    int32_t fresh;
    pa_status st = pa_alloc_block(a, &fresh);
    if (st != PA_OK) return st;
    a->ref[block] -= 1;
    *new_block_out = fresh;
    *copied = 1;
    return PA_OK;
}

pa_status pa_alloc_append_slot(pa_allocator* a, int32_t* table_row, int32_t capacity,
                               int32_t* num_blocks, int32_t position, int32_t block_size,
                               int64_t* slot_out, int32_t* cow_src, int32_t* cow_dst) {
    if (a == nullptr || table_row == nullptr || num_blocks == nullptr || slot_out == nullptr ||
        cow_src == nullptr || cow_dst == nullptr || block_size <= 0 || capacity < 0)
        return PA_ERR_INVALID;
    const int32_t n = *num_blocks;
    if (n < 0 || n > capacity) return PA_ERR_INVALID;
    if (position < 0 || static_cast<int64_t>(position) > static_cast<int64_t>(n) * block_size)
        return PA_ERR_RANGE;
    const int32_t j = position / block_size;
    int32_t src = -1, dst = -1;
    if (j == n) {  // the sequence's blocks are full: take a new one
        if (j >= capacity) return PA_ERR_RANGE;
        int32_t b;
        pa_status st = pa_alloc_block(a, &b);
        if (st != PA_OK) return st;
        table_row[j] = b;
        *num_blocks = n + 1;
    } else {  // writing into an existing block: private copy if it is shared
        int32_t b = table_row[j];
        int32_t fresh, copied;
        pa_status st = pa_alloc_cow(a, b, &fresh, &copied);
        if (st != PA_OK) return st;
        if (copied) {
            table_row[j] = fresh;
            src = b;
            dst = fresh;
        }
    }
    *slot_out = static_cast<int64_t>(table_row[j]) * block_size + position % block_size;
    *cow_src = src;
    *cow_dst = dst;
    return PA_OK;
}

pa_status pa_alloc_fork(pa_allocator* a, const int32_t* table_row, int32_t num_blocks) {
    if (a == nullptr || (table_row == nullptr && num_blocks > 0) || num_blocks < 0) return PA_ERR_INVALID;
    for (int32_t i = 0; i < num_blocks; ++i) {
        pa_status st = pa_alloc_incref(a, table_row[i]);
        if (st != PA_OK) {
            for (int32_t k = i - 1; k >= 0; --k) a->ref[table_row[k]] -= 1;  // were >= 2
            return st;
        }
    }
    return PA_OK;
}

pa_status pa_alloc_free_sequence(pa_allocator* a, const int32_t* table_row, int32_t num_blocks) {
    if (a == nullptr || (table_row == nullptr && num_blocks > 0) || num_blocks < 0) return PA_ERR_INVALID;
    // validate first so that a failure leaves the state unchanged: every id in
    // range and each block referenced at least as often as the row names it
    std::unordered_map<int32_t, int32_t> uses;
    for (int32_t i = 0; i < num_blocks; ++i) {
        int32_t b = table_row[i];
        if (!valid_id(a, b)) return PA_ERR_RANGE;
        if (a->ref[b] < ++uses[b]) return PA_ERR_INVALID;
    }
    for (int32_t i = 0; i < num_blocks; ++i) pa_alloc_decref(a, table_row[i]);
    return PA_OK;
}

pa_status pa_alloc_truncate(pa_allocator* a, int32_t* table_row, int32_t capacity, int32_t* num_blocks,
                            int32_t* start, int32_t* length, int32_t keep, int32_t block_size) {
    if (a == nullptr || table_row == nullptr || num_blocks == nullptr || start == nullptr || length == nullptr ||
        block_size <= 0)
        return PA_ERR_INVALID;
    const int32_t nb = *num_blocks, st = *start, len = *length;
    if (keep < 0 || nb < 0 || nb > capacity || st < 0 || st > len ||
        static_cast<int64_t>(len) > static_cast<int64_t>(nb) * block_size)
        return PA_ERR_RANGE;
    // the new first position; every block wholly before it goes back to the pool
    const int32_t new_start = std::max(st, len - std::min(keep, len));
    const int32_t drop = new_start / block_size;
    std::unordered_map<int32_t, int32_t> uses;
    for (int32_t i = 0; i < drop; ++i) {
        const int32_t b = table_row[i];
        if (!valid_id(a, b)) return PA_ERR_RANGE;
        if (a->ref[b] < ++uses[b]) return PA_ERR_INVALID;
    }
    for (int32_t i = 0; i < drop; ++i) pa_alloc_decref(a, table_row[i]);
    for (int32_t i = 0; i + drop < nb; ++i) table_row[i] = table_row[i + drop];
    for (int32_t i = nb - drop; i < nb; ++i) table_row[i] = -1;
    *num_blocks = nb - drop;
    *start = new_start - drop * block_size;
    *length = len - drop * block_size;
    return PA_OK;
}

pa_status pa_alloc_dump(const pa_allocator* a, int32_t* free_stack_out, int32_t* free_count_out,
                        int32_t* refcounts_out) {
    if (a == nullptr || free_stack_out == nullptr || free_count_out == nullptr || refcounts_out == nullptr)
        return PA_ERR_INVALID;
    const size_t nf = a->free_stack.size();
    for (size_t i = 0; i < nf; ++i) free_stack_out[i] = a->free_stack[i];
    *free_count_out = static_cast<int32_t>(nf);
    for (int32_t i = 0; i < a->num_blocks; ++i) refcounts_out[i] = a->ref[i];
    return PA_OK;
}

}  // extern "C"
