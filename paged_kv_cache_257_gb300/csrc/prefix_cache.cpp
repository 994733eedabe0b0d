// Automatic prefix caching: a hash table of full KV blocks keyed by prefix.
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 5, 2 "Automatic Prefix Caching": a new
// request whose tokens match a previously computed sequence has the matching
// physical blocks looked up in a hash table and mapped into its block table,
// so their prefill is skipped and the shared prefix takes no new memory.
// hyperinfer.ai "KV cache & paged attention deep dive", "Prefix caching:
// share the system prompt": one copy of the prefix KV for every request.
//
// The pages name no hash and no policy.  Block j of a token sequence is keyed
// by FNV-1a-64 (Fowler-Noll-Vo) over the little-endian bytes of the previous
// block's key (0 before block 0) followed by the block's token ids as 32-bit
// values, so a key stands for the whole prefix up to its block.  Hits are
// verified against the stored parent key and tokens; the cache holds one
// reference per cached block; eviction releases blocks only the cache still
// references, least recently used first, deeper blocks first within one use.
#include <algorithm>
#include <cstdint>
#include <new>
#include <tuple>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "pagedattn.h"

namespace {

constexpr uint64_t kFnvOffset = 0xcbf29ce484222325ULL;
constexpr uint64_t kFnvPrime = 0x100000001b3ULL;

inline uint64_t fnv_byte(uint64_t h, uint8_t b) { return (h ^ b) * kFnvPrime; }

uint64_t block_key(uint64_t parent, const int32_t* tokens, int32_t n) {
    uint64_t h = kFnvOffset;
    for (int i = 0; i < 8; ++i) h = fnv_byte(h, static_cast<uint8_t>(parent >> (8 * i)));
    for (int32_t t = 0; t < n; ++t) {
        const uint32_t v = static_cast<uint32_t>(tokens[t]);
        for (int i = 0; i < 4; ++i) h = fnv_byte(h, static_cast<uint8_t>(v >> (8 * i)));
    }
    return h;
}

struct Entry {
    int32_t block;
    uint64_t parent;
    std::vector<int32_t> tokens;
    int32_t depth;
    int64_t tick;
    int64_t order;
};

}  // namespace

struct pa_prefix_cache {
    pa_allocator* alloc;
    int32_t block_size;
    std::unordered_map<uint64_t, Entry> entries;
    std::unordered_set<int32_t> cached_blocks;
    int64_t tick = 0;
    int64_t order = 0;

    bool same(const Entry& e, uint64_t parent, const int32_t* toks) const {
        return e.parent == parent && std::equal(e.tokens.begin(), e.tokens.end(), toks);
    }
};

extern "C" {

uint64_t pa_prefix_block_key(uint64_t parent_key, const int32_t* tokens, int32_t num_tokens) {
    if (tokens == nullptr || num_tokens < 0) return 0;
    return block_key(parent_key, tokens, num_tokens);
}

pa_status pa_prefix_create(pa_allocator* alloc, int32_t block_size, pa_prefix_cache** out) {
    if (out == nullptr) return PA_ERR_INVALID;
    *out = nullptr;
    if (alloc == nullptr || block_size <= 0) return PA_ERR_INVALID;
    pa_prefix_cache* c = new (std::nothrow) pa_prefix_cache();
    if (c == nullptr) return PA_ERR_OOM;
    c->alloc = alloc;
    c->block_size = block_size;
    *out = c;
    return PA_OK;
}

void pa_prefix_destroy(pa_prefix_cache* c) {
    if (c == nullptr) return;
    std::vector<const Entry*> all;
    all.reserve(c->entries.size());
    for (const auto& kv : c->entries) all.push_back(&kv.second);
    std::sort(all.begin(), all.end(), [](const Entry* x, const Entry* y) { return x->order < y->order; });
    for (const Entry* e : all) pa_alloc_decref(c->alloc, e->block);
    delete c;
}

int32_t pa_prefix_size(const pa_prefix_cache* c) {
    return c == nullptr ? -1 : static_cast<int32_t>(c->entries.size());
}

pa_status pa_prefix_match(pa_prefix_cache* c, const int32_t* tokens, int32_t num_tokens, int32_t* table_row,
                          int32_t capacity, int32_t* matched_blocks) {
    if (c == nullptr || matched_blocks == nullptr || num_tokens < 0 || capacity < 0 ||
        (tokens == nullptr && num_tokens > 0) || (table_row == nullptr && capacity > 0))
        return PA_ERR_INVALID;
    ++c->tick;
    const int32_t bs = c->block_size;
    const int32_t n = std::min(num_tokens / bs, capacity);
    uint64_t parent = 0;
    int32_t m = 0;
    for (int32_t j = 0; j < n; ++j) {
        const int32_t* blk = tokens + static_cast<int64_t>(j) * bs;
        const uint64_t key = block_key(parent, blk, bs);
        auto it = c->entries.find(key);
        if (it == c->entries.end() || !c->same(it->second, parent, blk)) break;
        if (pa_alloc_incref(c->alloc, it->second.block) != PA_OK) break;   // cannot fail: the cache holds it
        table_row[j] = it->second.block;
        it->second.tick = c->tick;
        ++m;
        parent = key;
    }
    *matched_blocks = m;
    return PA_OK;
}

pa_status pa_prefix_insert(pa_prefix_cache* c, const int32_t* tokens, int32_t num_tokens, const int32_t* table_row,
                           int32_t num_blocks, int32_t* inserted) {
    if (c == nullptr || inserted == nullptr || num_tokens < 0 || num_blocks < 0 ||
        (tokens == nullptr && num_tokens > 0) || (table_row == nullptr && num_blocks > 0))
        return PA_ERR_INVALID;
    *inserted = 0;
    const int32_t bs = c->block_size;
    const int32_t n = std::min(num_blocks, num_tokens / bs);
    // plan first, so that a bad id changes nothing
    struct Step {
        bool fresh;
        uint64_t key;
        Entry e;
    };
    std::vector<Step> plan;
    std::unordered_map<uint64_t, size_t> planned;   // key -> index in plan (fresh entries)
    std::unordered_set<int32_t> planned_blocks;
    uint64_t parent = 0;
    for (int32_t j = 0; j < n; ++j) {
        const int32_t* blk = tokens + static_cast<int64_t>(j) * bs;
        const uint64_t key = block_key(parent, blk, bs);
        const Entry* e = nullptr;
        auto it = c->entries.find(key);
        if (it != c->entries.end()) {
            e = &it->second;
        } else {
            auto pt = planned.find(key);
            if (pt != planned.end()) e = &plan[pt->second].e;
        }
        if (e != nullptr) {
            if (!c->same(*e, parent, blk)) break;   // collision: the owner's chain stays
            plan.push_back({false, key, Entry{}});
            parent = key;
            continue;
        }
        const int32_t b = table_row[j];
        if (c->cached_blocks.count(b) || planned_blocks.count(b)) break;   // one key per block
        const int32_t r = pa_alloc_refcount(c->alloc, b);
        if (r < 0) return PA_ERR_RANGE;
        if (r == 0) return PA_ERR_INVALID;
        Entry ne{b, parent, std::vector<int32_t>(blk, blk + bs), j, 0, 0};
        planned[key] = plan.size();
        planned_blocks.insert(b);
        plan.push_back({true, key, std::move(ne)});
        parent = key;
    }
    ++c->tick;
    int32_t made = 0;
    for (Step& s : plan) {
        if (!s.fresh) {
            c->entries[s.key].tick = c->tick;
            continue;
        }
        pa_alloc_incref(c->alloc, s.e.block);
        s.e.tick = c->tick;
        s.e.order = c->order++;
        c->cached_blocks.insert(s.e.block);
        c->entries.emplace(s.key, std::move(s.e));
        ++made;
    }
    *inserted = made;
    return PA_OK;
}

pa_status pa_prefix_evict(pa_prefix_cache* c, int32_t max_blocks, int32_t* evicted) {
    if (c == nullptr || evicted == nullptr) return PA_ERR_INVALID;
    *evicted = 0;
    std::vector<std::tuple<int64_t, int32_t, uint64_t>> cands;   // (tick, -depth, key)
    for (const auto& kv : c->entries)
        if (pa_alloc_refcount(c->alloc, kv.second.block) == 1)
            cands.emplace_back(kv.second.tick, -kv.second.depth, kv.first);
    std::sort(cands.begin(), cands.end());
    const size_t n = std::min(cands.size(), static_cast<size_t>(std::max(max_blocks, 0)));
    for (size_t i = 0; i < n; ++i) {
        auto it = c->entries.find(std::get<2>(cands[i]));
        const int32_t b = it->second.block;
        c->entries.erase(it);
        c->cached_blocks.erase(b);
        pa_alloc_decref(c->alloc, b);
    }
    *evicted = static_cast<int32_t>(n);
    return PA_OK;
}

}  // extern "C"
