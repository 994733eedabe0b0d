// Entry points of decode attention: argument checks, partition choice,
// workspace layout and kernel dispatch.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

#include "decode.h"
#include "pagedattn.h"

namespace pa {
namespace {

constexpr int kMaxParts = 32768;

std::atomic<int32_t> g_deterministic{0};   // pa_set_decode_deterministic
std::atomic<int32_t> g_kernel{PA_DECODE_KERNEL_AUTO};   // pa_set_decode_kernel

// Workspace layout of a split call: merge tickets, partial outputs and
// partial (max, sum) pairs.  An unsplit call needs none.
struct WorkspaceLayout {
    size_t tickets_bytes, part_o_bytes, part_ml_bytes;
    size_t total() const { return tickets_bytes + part_o_bytes + part_ml_bytes; }
};

WorkspaceLayout layout(const pa_cache_desc* c, int64_t batch, int64_t num_q_heads, int64_t parts) {
    const int64_t groups = (num_q_heads / c->num_kv_heads + kHeadsPerCta - 1) / kHeadsPerCta;
    WorkspaceLayout w{};
    if (parts <= 1) return w;
    w.tickets_bytes = (static_cast<size_t>(batch * c->num_kv_heads * groups) * sizeof(int32_t) + 255) / 256 * 256;
    w.part_o_bytes = static_cast<size_t>(batch * num_q_heads * parts * c->head_dim) * sizeof(float);
    w.part_ml_bytes = static_cast<size_t>(batch * num_q_heads * parts * 2) * sizeof(float);
    return w;
}

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

// Tokens per partition must be a multiple of the 16-token chunk and of the block size.
int32_t partition_unit(int32_t block_size) { return std::max(16, block_size); }

// Partition planning.  A work item (one CTA) covers one partition of one
// sequence for one group of query heads; the resident CTAs stream the KV
// cache at a shared rate, so a call takes about
//     waves x (tokens of the longest item + kItemOverheadTokens)
// with waves = ceil(items / resident CTAs).  The overhead stands for what an
// item costs beyond its tokens (filling and draining its pipeline, writing
// and merging a partial); 192 tokens matches the partition sweeps of the
// tensor-core kernel on GB300 (Llama-3-8B ragged batch, 13B MHA, 70B 128k FP8).
constexpr int64_t kItemOverheadTokens = 192;

int64_t plan_cost(int64_t items, int64_t longest_item, int64_t slots) {
    const int64_t waves = std::max<int64_t>(1, (items + slots - 1) / slots);
    return waves * (longest_item + kItemOverheadTokens);
}

// The partition with the least modelled time among the whole context, the
// powers of two from 8192 down to 256 tokens and, where their items fit one
// wave, the multiples of 128 between 1024 and 4096 (first come, first kept
// on ties: the powers of two and the larger partitions, which leave fewer
// partials).  The finer grid lets a batch of long items fill one wave: 64
// sequences of 2049 to 2561 tokens (the prefix-sharing workload) take
// 2304-token partitions, half of them split in two, and decode in 43.9 us
// against 49.8 us whole.  Finer steps measured slower below 1024 tokens (a
// 1000-token window of the Llama-3-8B batch: 384-token partitions 25.7 us
// against 24.8 at 512) and over two waves (4 x 131072 FP8 tokens: 2816-token
// partitions 169.6 us against 166.2 at 2048).
// `lens` holds the batch's context lengths, or is null to assume every
// sequence at `cap`.
int32_t plan_partition(const pa_cache_desc* c, int32_t batch, int32_t num_q_heads, int64_t cap,
                       const int32_t* lens, int32_t num_sms) {
    const int32_t unit = partition_unit(c->block_size);
    const int64_t groups = (num_q_heads / c->num_kv_heads + kHeadsPerCta - 1) / kHeadsPerCta;
    const int64_t per_seq = static_cast<int64_t>(c->num_kv_heads) * groups;
    const int64_t slots = static_cast<int64_t>(PA_DECODE_MIN_CTAS) * std::max(num_sms, 1);
    const int64_t whole = std::max<int64_t>((cap + unit - 1) / unit * unit, unit);
    // items (partitions x head groups) and the longest partition share for a
    // partition size p: a sequence of len tokens splits into ceil(len / p)
    // equal shares, each rounded up to the unit
    auto model = [&](int64_t p, int64_t& items, int64_t& longest) {
        items = 0;
        longest = 0;
        for (int32_t s = 0; s < batch; ++s) {
            const int64_t len = lens ? std::min<int64_t>(std::max(lens[s], 0), cap) : cap;
            if (len == 0) continue;
            const int64_t n = (len + p - 1) / p;
            const int64_t share = ((len + n - 1) / n + unit - 1) / unit * unit;
            items += n;
            longest = std::max(longest, std::min(share, len));
        }
        items *= per_seq;
    };
    int64_t items = 0, longest = 0;
    model(whole, items, longest);
    int64_t best = whole;
    int64_t best_cost = plan_cost(items, longest, slots);
    auto consider = [&](int64_t p, bool one_wave_only) {
        if (p % unit != 0 || p >= whole) return;
        model(p, items, longest);
        if (one_wave_only && items > slots) return;
        const int64_t cost = plan_cost(items, longest, slots);
        if (cost < best_cost) {
            best = p;
            best_cost = cost;
        }
    };
    for (int64_t p = 8192; p >= 256; p /= 2) consider(p, false);
    for (int64_t p = 4096 - 128; p > 1024; p -= 128)
        if ((p & (p - 1)) != 0) consider(p, true);
    return static_cast<int32_t>(best);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" int32_t pa_decode_partition_size(const pa_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                            int32_t max_blocks_per_seq, int32_t requested) {
    if (check_cache_desc(cache) != PA_OK || batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 ||
        num_q_heads % cache->num_kv_heads != 0)
        return -1;
    const int32_t unit = partition_unit(cache->block_size);
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * cache->block_size;
    if (cap >= (int64_t{1} << 31)) return -1;
    if (requested == -1) return static_cast<int32_t>((cap + unit - 1) / unit * unit);
    if (requested > 0) return requested % unit == 0 ? requested : -1;
    if (requested == 0) return plan_partition(cache, batch, num_q_heads, cap, nullptr, sm_count());
    return -1;
}

extern "C" int32_t pa_decode_plan_partition(const pa_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                            int32_t max_blocks_per_seq, const int32_t* host_context_lens,
                                            int32_t num_sms) {
    if (check_cache_desc(cache) != PA_OK || batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 ||
        num_q_heads % cache->num_kv_heads != 0)
        return -1;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * cache->block_size;
    if (cap >= (int64_t{1} << 31)) return -1;
    if (num_sms <= 0) num_sms = sm_count();
    if (num_sms <= 0) return -1;
    return plan_partition(cache, batch, num_q_heads, cap, host_context_lens, num_sms);
}

namespace pa {

size_t decode_counter_bytes(const pa_cache_desc* c, int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                            int32_t partition_size) {
    const int32_t p = pa_decode_partition_size(c, batch, num_q_heads, max_blocks, partition_size);
    if (p <= 0) return 0;
    const int64_t cap = static_cast<int64_t>(max_blocks) * c->block_size;
    const WorkspaceLayout w = layout(c, batch, num_q_heads, (cap + p - 1) / p);
    return w.tickets_bytes;
}

// Kernel choice for the tensor-core path.  One warp streams an item about
// four times slower than a CTA of four warps, but it pays no pipeline fill
// of its own while other warps stream and no cross-warp merge; that wins
// when the items are long (partitions of 512 tokens or more) and many.  The
// host does not know the context lengths (or window starts) here, so the
// count is the grid's upper bound, every sequence at the table's capacity,
// and it must cover two waves of warp slots (counted at 20 per SM, the FP8
// residency, for every cache type).  Measured on GB300 (decode us,
// CTA kernel / warp kernel, upper bound on items): 128k-token FP8 contexts
// in 512-token partitions 175 / 165 (8192); their last 32760 tokens
// 56.5 / 51.4 (8192, 2048 real); a Llama-3-8B ragged batch in 512-token
// partitions 49.0 / 48.5 (2048), the same batch's last 1000 tokens
// 24.9 / 30.8 (2048, about 512 real).
bool warp_path_preferred(const DecodeArgs& a) {
    if (a.partition_size < 512) return false;
    const int64_t n_hg = (a.group + kHeadsPerCta - 1) / kHeadsPerCta;
    const int64_t items = static_cast<int64_t>(a.max_parts) * a.num_kv_heads * n_hg * a.batch;
    const int64_t slots = static_cast<int64_t>(PA_DECODE_WARP_MIN_CTAS) * std::max(sm_count(), 1);
    return items >= 2 * slots;
}

}  // namespace pa

extern "C" size_t pa_decode_workspace_size(const pa_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                           int32_t max_blocks_per_seq, int32_t partition_size) {
    const int32_t p = pa_decode_partition_size(cache, batch, num_q_heads, max_blocks_per_seq, partition_size);
    if (p <= 0) return 0;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * cache->block_size;
    return layout(cache, batch, num_q_heads, (cap + p - 1) / p).total();
}

extern "C" pa_status pa_decode_attention_window(const pa_cache_desc* cache, const void* q, pa_dtype q_dtype,
                                                int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                const int32_t* context_lens, const int32_t* context_starts,
                                                int32_t batch, float scale, int32_t partition_size, void* workspace,
                                                size_t workspace_bytes, void* out, pa_dtype out_dtype,
                                                int32_t* device_status, void* stream_) {
    pa_status st = check_cache_desc(cache);
    if (st != PA_OK) return st;
    if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0) return PA_ERR_INVALID;
    if (num_q_heads % cache->num_kv_heads != 0) return PA_ERR_INVALID;
    if (q_dtype != PA_F32 && q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (out_dtype != PA_F32 && out_dtype != PA_F16 && out_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
    if (!std::isfinite(scale)) return PA_ERR_INVALID;
    if (batch == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(context_starts, 4) ||
        !aligned(device_status, 4) || !aligned(workspace, 16))
        return PA_ERR_INVALID;
    const int32_t group = num_q_heads / cache->num_kv_heads;
    const int64_t n_hg = (group + kHeadsPerCta - 1) / kHeadsPerCta;
    if (batch > 65535 || cache->num_kv_heads * n_hg > 65535) return PA_ERR_UNSUPPORTED;
    const int64_t cap = static_cast<int64_t>(max_blocks_per_seq) * cache->block_size;
    if (cap >= (int64_t{1} << 31)) return PA_ERR_UNSUPPORTED;

    const int32_t p = pa_decode_partition_size(cache, batch, num_q_heads, max_blocks_per_seq, partition_size);
    if (p <= 0) return PA_ERR_INVALID;
    const int64_t parts = (cap + p - 1) / p;
    if (parts > kMaxParts) return PA_ERR_UNSUPPORTED;
    const size_t need = pa_decode_workspace_size(cache, batch, num_q_heads, max_blocks_per_seq, p);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return PA_ERR_INVALID;

    DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.context_starts = context_starts;
    a.out = out;
    const WorkspaceLayout wl = layout(cache, batch, num_q_heads, parts);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const bool split = wl.tickets_bytes > 0;
    a.tickets = split ? reinterpret_cast<int32_t*>(ws) : nullptr;
    a.part_o = split ? reinterpret_cast<float*>(ws + wl.tickets_bytes) : nullptr;
    a.part_ml = split ? reinterpret_cast<float*>(ws + wl.tickets_bytes + wl.part_o_bytes) : nullptr;
    a.fused_merge = parts <= kFusedMergeMaxParts ? 1 : 0;
    a.balanced_tail = g_deterministic.load(std::memory_order_relaxed) ? 0 : 1;
    a.status = device_status;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = cache->num_kv_heads;
    a.head_dim = cache->head_dim;
    a.block_size = cache->block_size;
    a.num_blocks = cache->num_blocks;
    a.max_blocks = max_blocks_per_seq;
    a.group = group;
    a.partition_size = p;
    a.max_parts = static_cast<int32_t>(parts);
    a.q_dtype = q_dtype;
    a.kv_dtype = cache->kv_dtype;
    a.out_dtype = out_dtype;
    a.scale = scale;
    a.k_scale = cache->kv_dtype == PA_FP8_E4M3 ? cache->k_scale : 1.f;
    a.v_scale = cache->kv_dtype == PA_FP8_E4M3 ? cache->v_scale : 1.f;

    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    if (!mma_path_supported(a))
        st = launch_decode_simt(a, s);
    else {
        const int32_t k = g_kernel.load(std::memory_order_relaxed);
        const bool warp = k == PA_DECODE_KERNEL_WARP || (k == PA_DECODE_KERNEL_AUTO && warp_path_preferred(a));
        st = warp ? launch_decode_warp(a, s) : launch_decode_mma(a, s);
    }
    if (st == PA_OK && parts > 1 && !a.fused_merge) st = launch_decode_reduce(a, s);
    return st;
}

extern "C" pa_status pa_decode_attention(const pa_cache_desc* cache, const void* q, pa_dtype q_dtype,
                                         int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* context_lens, int32_t batch, float scale,
                                         int32_t partition_size, void* workspace, size_t workspace_bytes,
                                         void* out, pa_dtype out_dtype, int32_t* device_status, void* stream) {
    return pa_decode_attention_window(cache, q, q_dtype, num_q_heads, k_cache, v_cache, block_tables,
                                      max_blocks_per_seq, context_lens, nullptr, batch, scale, partition_size,
                                      workspace, workspace_bytes, out, out_dtype, device_status, stream);
}

extern "C" void pa_set_decode_deterministic(int32_t on) { g_deterministic.store(on ? 1 : 0, std::memory_order_relaxed); }

extern "C" int32_t pa_get_decode_deterministic(void) { return g_deterministic.load(std::memory_order_relaxed); }

extern "C" pa_status pa_set_decode_kernel(int32_t kernel) {
    if (kernel != PA_DECODE_KERNEL_AUTO && kernel != PA_DECODE_KERNEL_CTA && kernel != PA_DECODE_KERNEL_WARP)
        return PA_ERR_INVALID;
    g_kernel.store(kernel, std::memory_order_relaxed);
    return PA_OK;
}

extern "C" int32_t pa_get_decode_kernel(void) { return g_kernel.load(std::memory_order_relaxed); }
