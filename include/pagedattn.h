/* pagedattn.h - C ABI of the GB300 paged decode-attention library.
 *
 * The library implements the decode hot path of PagedAttention as the pages
 * describe it: the KV cache of every sequence lives in fixed-size physical
 * blocks drawn from one pre-allocated pool and is reached through a
 * per-sequence block table; each decode step appends the new token's K and V
 * to its slot and computes single-query attention softmax(q K^T * scale) V
 * over the sequence's cached tokens.
 *
 * Pages cited (title, section):
 *   [DEV] dev.to/syed_anzar, "Why LLMs Run Out of VRAM: KV Cache Fragmentation
 *         and How PagedAttention Fixes It"
 *   [HI]  hyperinfer.ai, "KV cache & paged attention deep dive"
 *   [VK]  vaibhawkumar.in, "Why LLMs run out of VRAM: KV cache fragmentation and
 *         the PagedAttention fix"
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses owned by the caller; the
 *     library never allocates, frees or retains device memory.  Host
 *     pointers are plain host memory owned by the caller.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Device work is enqueued asynchronously on it.
 *   - Every call returns a pa_status; no exception or abort crosses the ABI.
 *     Arguments are validated on the host before anything is enqueued; an
 *     invalid call enqueues nothing.
 *   - Values that live in device memory (slots, block ids, context lengths)
 *     cannot be checked on the host.  Kernels check them and never read or
 *     write outside the buffers described by the arguments: a bad value
 *     sets a bit of the optional `device_status` word (a device int32 the
 *     caller zeroes; NULL disables reporting) and the affected element is
 *     skipped or clamped.  Results of a call that raised a device flag are
 *     unspecified.  pa_read_device_status() reads the word back.
 *   - Device kernels never trap and never wait without a time limit; a
 *     wait that runs out sets PA_DEVFLAG_TIMEOUT and the kernel returns.
 *     When PA_DEVFLAG_TIMEOUT is set, the whole output of that call is
 *     undefined (not only the rows whose wait ran out: a CTA that gave up
 *     may reuse on-chip buffers that late copies still land in).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,      /* bad argument: null pointer, bad size, misaligned buffer */
    PA_ERR_OOM = 2,          /* block allocator: the free pool is empty                 */
    PA_ERR_RANGE = 3,        /* block id, position or slot outside its range            */
    PA_ERR_UNSUPPORTED = 4,  /* well-formed but not implemented (head_dim, dtype pair)  */
    PA_ERR_CUDA = 5,         /* a CUDA runtime or driver call failed                    */
    PA_ERR_DEVICE_FLAG = 6   /* pa_read_device_status found a raised device flag        */
} pa_status;

/* Element types.  PA_FP8_E4M3 is the OCP 8-bit E4M3 format without
 * infinities (max +-448); a cache of this type stores round-to-nearest-even,
 * saturating codes of x / scale and is read back as code * scale. */
typedef enum pa_dtype { PA_F32 = 0, PA_F16 = 1, PA_BF16 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

/* Bits of the device status word. */
#define PA_DEVFLAG_SLOT_RANGE    1  /* append: slot < 0 or >= num_blocks*block_size (row skipped) */
#define PA_DEVFLAG_BLOCK_RANGE   2  /* decode: block-table entry outside [0, num_blocks)            */
#define PA_DEVFLAG_CONTEXT_RANGE 4  /* decode: context_len < 0 or > max_blocks_per_seq*block_size */
#define PA_DEVFLAG_TIMEOUT       8  /* a bounded on-chip wait ran out                               */

/* One paged KV cache (one layer): two pools, K and V, each laid out
 *   [num_blocks][num_kv_heads][block_size][head_dim]
 * contiguous, so the block_size x head_dim tokens of one (physical block,
 * KV head) pair are one run of memory.  Token slot s lives in physical block
 * s / block_size at offset s % block_size.  [DEV] section 4 "How the
 * Architecture Works" (fixed-size blocks in one pool, block tables); the
 * pool layout itself is this library's choice.
 *   block_size : tokens per block, 8, 16 or 32 ([DEV] section 6 "Select the
 *                Right Block Size": 16 by default, 32 an option)
 *   head_dim   : 64, 128 or 256
 *   k_scale, v_scale : PA_FP8_E4M3 only, the float32 dequantisation scale of
 *                each pool (one per cache tensor); ignored otherwise. */
typedef struct pa_cache_desc {
    int32_t num_blocks;
    int32_t block_size;
    int32_t num_kv_heads;
    int32_t head_dim;
    pa_dtype kv_dtype;
    float k_scale;
    float v_scale;
} pa_cache_desc;

/* ---------------------------------------------------------------- misc */

/* Library version string (static storage). */
const char* pa_version(void);

/* Human-readable name of a status (static storage). */
const char* pa_status_string(pa_status status);

/* Bytes of one element of `dtype`; 0 for an unknown type. */
size_t pa_dtype_size(pa_dtype dtype);

/* KV-cache bytes per token over a whole model: 2 * n_layers * n_kv_heads *
 * head_dim * sizeof(dtype).  [DEV] section 2 "The Concrete Math of KV Cache
 * Growth" (Example 1: 819,200 B; Example 2: 131,072 B); [HI] "What the KV
 * cache is, and why it dominates memory".  Returns 0 for negative sizes or
 * an unknown dtype. */
uint64_t pa_kv_bytes_per_token(int32_t n_layers, int32_t n_kv_heads, int32_t head_dim, pa_dtype dtype);

/* ------------------------------------------------------ slot mapping */

/* Host computation of the slot each new token is written to:
 *   slots_out[t] = block_tables[seq_ids[t]][positions[t] / block_size] * block_size
 *                  + positions[t] % block_size
 * [DEV] section 4 "How the Architecture Works": the block table holds the
 * physical block of each logical block.  All pointers are HOST memory:
 *   block_tables [batch][max_blocks] int32, seq_ids [num_tokens] int32,
 *   positions [num_tokens] int32, slots_out [num_tokens] int64 (written).
 * PA_ERR_RANGE if a sequence id is outside [0, batch), a position is
 * negative or past the table (nothing is written then); PA_ERR_INVALID for
 * null pointers or non-positive sizes (num_tokens == 0 is a no-op). */
pa_status pa_compute_slot_mapping(const int32_t* block_tables, int32_t batch, int32_t max_blocks,
                                  int32_t block_size, const int32_t* seq_ids,
                                  const int32_t* positions, int32_t num_tokens, int64_t* slots_out);

/* ----------------------------------------------------------- KV append */

/* Write each new token's K and V rows into the slot slot_mapping[t] names.
 * [DEV] section 1 "Why Transformers Need a KV Cache" (append the new
 * token's K and V each step) and section 4 (into the block the table
 * names); [VK] "A minimal PyTorch sketch" (append writes rows into the
 * current page).
 *   k, v          device [num_tokens][num_kv_heads][head_dim] of src_dtype
 *   slot_mapping  device [num_tokens] int64
 *   k_cache, v_cache  device pools of cache->kv_dtype (layout above)
 * Type pairs (src -> cache): same type (bit copy); PA_F32 -> PA_F16 / PA_BF16
 * (round to nearest even); PA_F32 / PA_F16 / PA_BF16 -> PA_FP8_E4M3 (the
 * float32 value divided by k_scale / v_scale in IEEE float32, then rounded
 * to nearest even E4M3 with saturation to +-448).  Others: PA_ERR_UNSUPPORTED.
 * A slot outside [0, num_blocks*block_size) skips that token and sets
 * PA_DEVFLAG_SLOT_RANGE.  Duplicate slots in one call leave either row.
 * Buffers must be 16-byte aligned. */
pa_status pa_kv_append(const pa_cache_desc* cache, const void* k, const void* v, pa_dtype src_dtype,
                       const int64_t* slot_mapping, int32_t num_tokens, void* k_cache, void* v_cache,
                       int32_t* device_status, void* stream);

/* Copy whole physical blocks, K and V pools, every KV head: for i <
 * num_pairs, block dst_blocks[i] receives the contents of src_blocks[i].
 * This is the device half of copy-on-write ([DEV] section 5 "Zero-Copy
 * Forking": a branch writing into a shared block first gets a private copy).
 *   src_blocks, dst_blocks  device [num_pairs] int32
 * A pair with an id outside [0, num_blocks) is skipped and sets
 * PA_DEVFLAG_BLOCK_RANGE.  Pairs must not overlap (no block is both a source
 * and a destination in one call). */
pa_status pa_copy_blocks(const pa_cache_desc* cache, void* k_cache, void* v_cache,
                         const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                         int32_t* device_status, void* stream);

/* ------------------------------------------------ decode attention */

/* Tokens per split-context partition the library uses for this problem:
 * `requested` > 0 is checked (a multiple of 16 and of block_size) and
 * returned; 0 picks one as pa_decode_plan_partition does with every
 * sequence at max_blocks_per_seq*block_size tokens; -1 means one partition
 * covering that many tokens.  Returns -1 on invalid input. */
int32_t pa_decode_partition_size(const pa_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                 int32_t max_blocks_per_seq, int32_t requested);

/* Partition size for a batch whose context lengths the host knows (a
 * serving loop knows them: it built the block tables).  The pages do not
 * size partitions; this models a call as waves of work items (one per
 * partition, sequence and group of up to 8 query heads) over the resident
 * CTAs, each wave as long as its longest item plus a fixed per-item cost,
 * and returns the candidate (the whole context, the powers of two from 8192
 * down to 256 tokens, and the multiples of 128 between 1024 and 4096 whose
 * items fit one wave) with the least modelled time; ties keep the power of
 * two and the larger size.  Pass the result as pa_decode_attention's
 * partition_size with the same cache, batch, num_q_heads and
 * max_blocks_per_seq.
 *   host_context_lens  host [batch] int32 (null: every sequence full)
 *   num_sms            SMs to plan for; <= 0 asks the current device
 * Returns -1 on invalid input or when num_sms <= 0 and no device answers. */
int32_t pa_decode_plan_partition(const pa_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                 int32_t max_blocks_per_seq, const int32_t* host_context_lens,
                                 int32_t num_sms);

/* Bytes of device workspace pa_decode_attention needs for these arguments:
 * when contexts are split, the merge counters and the partial softmax state
 * of the partitions; 0 when every sequence fits one partition (or for
 * invalid input).  The workspace must be zero-filled before its first use;
 * every completed call leaves its counters at zero again, so one zeroed
 * buffer serves any sequence of calls that are not concurrent. */
size_t pa_decode_workspace_size(const pa_cache_desc* cache, int32_t batch, int32_t num_q_heads,
                                int32_t max_blocks_per_seq, int32_t partition_size);

/* Single-query paged decode attention for a batch of sequences:
 *   out[s][h] = sum_{t < ctx_s} softmax_t(scale * q[s][h] . K_s[t][h/G]) V_s[t][h/G]
 * with G = num_q_heads / num_kv_heads (query head h reads KV head h / G),
 * K_s / V_s the sequence's cached tokens reached through its block table,
 * FP8 values dequantised as code * k_scale / v_scale.  [DEV] section 1
 * (attention formula), section 2 Example 2 (grouped-query heads), section 4
 * "The PagedAttention CUDA Kernel" (read the query, look up the block table,
 * fetch K and V from scattered blocks).  Long contexts are split into
 * partitions of at most `partition_size` tokens whose partial results are
 * merged by log-sum-exp: by the last partition's CTA when a sequence has at
 * most 16 partitions, otherwise by a second kernel.  A sequence of len tokens
 * splits into n = ceil(len / partition_size) partitions of equal share
 * (ceil(len / n) rounded up to 16 tokens, or to the block size if larger),
 * so the work items of a ragged batch stay alike in size; a length that is a
 * multiple of partition_size gives partitions of exactly that size.
 *   q              device [batch][num_q_heads][head_dim] of q_dtype
 *   block_tables   device [batch][max_blocks_per_seq] int32
 *   context_lens   device [batch] int32, cached tokens per sequence (0 gives
 *                  an all-zero output row)
 *   scale          softmax scale (1/sqrt(head_dim) for the usual attention)
 *   partition_size as in pa_decode_partition_size
 *   workspace      device buffer of at least pa_decode_workspace_size()
 *                  bytes; 16-byte aligned,
 *                  zero-filled before its first use; calls sharing one
 *                  workspace must not run concurrently
 *   out            device [batch][num_q_heads][head_dim] of out_dtype
 *                  (PA_F32, PA_F16 or PA_BF16)
 * Supported: head_dim 64/128/256; num_q_heads a multiple of num_kv_heads;
 * q_dtype PA_F32, PA_F16 or PA_BF16 (PA_F16/PA_BF16 queries with an FP8
 * cache must lie within the float16 range).  Tensor cores serve 16-bit and
 * FP8 caches with head_dim 128 and 16-bit queries; other cases run on CUDA
 * cores.  Results are reproducible bit for bit only in the deterministic
 * schedule (pa_set_decode_deterministic).
 * Errors: PA_ERR_INVALID (bad sizes or scale, null or misaligned pointers, a
 * workspace smaller than needed), PA_ERR_UNSUPPORTED (dtype pair, grid
 * limits), PA_ERR_CUDA (a launch failed). */
pa_status pa_decode_attention(const pa_cache_desc* cache, const void* q, pa_dtype q_dtype,
                              int32_t num_q_heads, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t batch, float scale,
                              int32_t partition_size, void* workspace, size_t workspace_bytes,
                              void* out, pa_dtype out_dtype, int32_t* device_status, void* stream);

/* pa_decode_attention over a slid window: sequence s attends only the
 * positions context_starts[s] .. context_lens[s] - 1 of its block-table row
 * ([VK] "PagedAttention: the idea" and "A minimal PyTorch sketch",
 * truncate: after the oldest pages go back to the allocator, the rest of the
 * drop is an offset into the first kept page; pa_alloc_truncate returns that
 * start and length).  Blocks wholly before a start are never read, so their
 * table entries may hold anything.
 *   context_starts  device [batch] int32 in [0, context_lens[s]], or null
 *                   (every start 0: the same as pa_decode_attention).  A
 *                   start outside that range is clamped into it and raises
 *                   PA_DEVFLAG_CONTEXT_RANGE; an empty window gives a zero row.
 * Every other argument, the workspace size and the partition size are those
 * of pa_decode_attention. */
pa_status pa_decode_attention_window(const pa_cache_desc* cache, const void* q, pa_dtype q_dtype,
                                     int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, const int32_t* context_starts, int32_t batch,
                                     float scale, int32_t partition_size, void* workspace, size_t workspace_bytes,
                                     void* out, pa_dtype out_dtype, int32_t* device_status, void* stream);

/* pa_decode_attention for callers that cannot allocate device memory (the
 * pages have no counterpart: this serves the library's users).  Some callers
 * cannot call cudaMalloc: code inside a host framework or server that owns
 * all device memory through its own allocator and forbids other allocations,
 * decode loops that must not stall every stream on cudaMalloc's implicit
 * device synchronisation, and deployments whose device footprint is fixed
 * up front.  This entry point takes the same arguments as
 * pa_decode_attention except the workspace: the split-context workspace is a
 * static array of PA_NOALLOC_SCRATCH_BYTES in device memory that every GPU
 * loading the library holds until the process exits.  It allocates nothing
 * and calls no allocating routine; the caller still passes every input and
 * output.
 *   - PA_ERR_RANGE when pa_decode_workspace_size() for these arguments
 *     exceeds PA_NOALLOC_SCRATCH_BYTES (use larger partitions, a smaller
 *     batch, or pa_decode_attention with a caller-owned workspace).
 *   - The first call on a device looks up the array's device address with
 *     that device current and zero-fills it, synchronising the device; make
 *     that first call before any stream capture.  The same set-up runs
 *     again on the first call after the device's context was destroyed
 *     (cudaDeviceReset), since the new context holds the array elsewhere.
 *   - PA_ERR_INVALID for a null input or output pointer when the call needs
 *     the array (every other check is pa_decode_attention's).
 *   - Every call on a device shares the one array, which keeps the previous
 *     call's contents; each call clears the merge counters it needs on its
 *     stream before the kernels.  Calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race on the array: serialise them. */
#define PA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

pa_status pa_decode_attention_noalloc(const pa_cache_desc* cache, const void* q, pa_dtype q_dtype,
                                      int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t batch, float scale,
                                      int32_t partition_size, void* out, pa_dtype out_dtype,
                                      int32_t* device_status, void* stream);

/* Chunk schedule of the tensor-core decode kernel, for every later decode
 * call of the process.  The pages have no counterpart: it is a property of
 * this kernel.  Default (0): with 16-bit caches the last 16 chunks of a work
 * item go to whichever of the CTA's warps is free, which balances the warps
 * (Llama-3-8B ragged batch about 3% faster).  A warp's softmax reference and
 * summation order then depend on timing, so two runs on the same inputs can
 * differ at the level of bf16 rounding of the probabilities (well inside the
 * documented tolerance, but not bit for bit).  1: every chunk goes to a
 * fixed warp; results are bit-reproducible.  FP8 caches and the CUDA-core
 * kernel always use fixed schedules.  Takes effect for calls made after it
 * returns (a process-wide setting; no synchronisation with calls in flight).
 * pa_get_decode_deterministic returns the current setting. */
void pa_set_decode_deterministic(int32_t on);
int32_t pa_get_decode_deterministic(void);

/* Which tensor-core decode kernel serves every later decode call of the
 * process.  The pages have no counterpart: both compute the same attention
 * (within the tolerances above) and differ only in how work items map to
 * warps.
 *   PA_DECODE_KERNEL_AUTO (default): the library picks per call: one warp
 *     per work item when partitions are at least 512 tokens and the grid
 *     (every sequence counted at max_blocks_per_seq * block_size tokens)
 *     holds at least two work items per warp slot of the GPU (20 per SM),
 *     else one CTA of four warps per work item.
 *   PA_DECODE_KERNEL_CTA: always a CTA of four warps per work item (an
 *     item's chunks split among the warps, whose states are merged).
 *   PA_DECODE_KERNEL_WARP: always one warp per work item.
 * Calls on the CUDA-core kernel are unaffected.  Process-wide, like
 * pa_set_decode_deterministic; PA_ERR_INVALID for another value.
 * pa_get_decode_kernel returns the current setting. */
#define PA_DECODE_KERNEL_AUTO 0
#define PA_DECODE_KERNEL_CTA 1
#define PA_DECODE_KERNEL_WARP 2
pa_status pa_set_decode_kernel(int32_t kernel);
int32_t pa_get_decode_kernel(void);

/* Wait for `stream`, copy the device status word to *flags_out (may be
 * NULL) and, if `reset` is non-zero, zero it.  Returns PA_ERR_DEVICE_FLAG
 * if any flag was set, PA_OK otherwise. */
pa_status pa_read_device_status(int32_t* device_status, int32_t* flags_out, int32_t reset, void* stream);

/* -------------------------------------------------- block allocator */

/* Host-side physical block pool with reference counts and copy-on-write.
 * [DEV] section 4 "How the Architecture Works" (one pre-allocated pool,
 * on-demand allocation when a block fills) and section 5 "Zero-Copy
 * Forking" (shared blocks carry a reference count; a branch's first write
 * into a shared block gets a private copy); [HI] "What 16-token blocks buy
 * you" (evicting a sequence frees its blocks to the pool).
 * The free pool is a LIFO stack.  A pool created with seed 0 hands out
 * blocks 0, 1, 2, ...; seed != 0 hands them out in a Fisher-Yates shuffle
 * of 0..num_blocks-1 driven by SplitMix64(seed) (i from n-1 down to 1:
 * j = next() mod (i+1), swap).  A block whose count reaches 0 is pushed on
 * top.  Not thread-safe: the caller serialises calls on one handle.  Any
 * failing call leaves the state unchanged. */
typedef struct pa_allocator pa_allocator;

/* New pool of `num_blocks` free blocks; *out receives the handle (caller owns
 * it, release with pa_alloc_destroy).  PA_ERR_INVALID if num_blocks <= 0. */
pa_status pa_alloc_create(int32_t num_blocks, uint64_t seed, pa_allocator** out);
void pa_alloc_destroy(pa_allocator* a);
int32_t pa_alloc_num_blocks(const pa_allocator* a);
int32_t pa_alloc_free_count(const pa_allocator* a);
/* Reference count of `block`, -1 if out of range. */
int32_t pa_alloc_refcount(const pa_allocator* a, int32_t block);

/* Pop a free block (count becomes 1).  PA_ERR_OOM when the pool is empty. */
pa_status pa_alloc_block(pa_allocator* a, int32_t* block_out);
/* One more table points at `block` (fork / prefix share).  PA_ERR_RANGE for a
 * bad id, PA_ERR_INVALID if the block is free. */
pa_status pa_alloc_incref(pa_allocator* a, int32_t block);
/* One table fewer points at `block`; at 0 it returns to the pool. */
pa_status pa_alloc_decref(pa_allocator* a, int32_t block);
/* Block to write instead of `block`: itself if its count is 1 (*copied = 0),
 * else a fresh block (*copied = 1, `block` loses one reference); the caller
 * then copies the block's device contents (pa_copy_blocks). */
pa_status pa_alloc_cow(pa_allocator* a, int32_t block, int32_t* new_block_out, int32_t* copied);

/* Slot for writing logical token `position` of one sequence.  `table_row`
 * (host, `capacity` entries) holds *num_blocks valid ids.  position ==
 * *num_blocks * block_size takes a new block (appended to the row,
 * *num_blocks incremented); a position inside a block whose count is above
 * 1 takes a private copy first (row entry replaced, *cow_src / *cow_dst set;
 * both are -1 when no copy is needed).  PA_ERR_RANGE for a negative
 * position, a gap, or a full row; PA_ERR_OOM if a block is needed and the
 * pool is empty. */
pa_status pa_alloc_append_slot(pa_allocator* a, int32_t* table_row, int32_t capacity,
                               int32_t* num_blocks, int32_t position, int32_t block_size,
                               int64_t* slot_out, int32_t* cow_src, int32_t* cow_dst);

/* incref (fork) / decref (free) every block of a row, in row order.  On error
 * the blocks already processed are rolled back. */
/* Slide a sequence's window so that only its last `keep` tokens stay
 * ([VK] "PagedAttention: the idea": the oldest page goes back to the
 * allocator; "A minimal PyTorch sketch", truncate: whole pages first, the
 * rest of the drop as an offset into the first kept page, no copy).  The
 * sequence occupies row positions [*start, *length) of `table_row` (host,
 * `capacity` entries, *num_blocks valid; position p lives in block
 * table_row[p / block_size] at offset p % block_size).  The new first
 * position is max(*start, *length - keep); every block wholly before it is
 * released (decref, row order) and removed from the front of the row, the
 * remaining ids move to the front and the freed tail entries become -1;
 * positions then count from the first remaining block, so *start ends below
 * block_size.  Pass *start and *length as pa_decode_attention_window's
 * context start and length, and *length as the next append position.
 * PA_ERR_RANGE for keep < 0 or an inconsistent window or an id out of
 * range, PA_ERR_INVALID for a block released more often than it is held;
 * on error nothing changes. */
pa_status pa_alloc_truncate(pa_allocator* a, int32_t* table_row, int32_t capacity, int32_t* num_blocks,
                            int32_t* start, int32_t* length, int32_t keep, int32_t block_size);

pa_status pa_alloc_fork(pa_allocator* a, const int32_t* table_row, int32_t num_blocks);
pa_status pa_alloc_free_sequence(pa_allocator* a, const int32_t* table_row, int32_t num_blocks);

/* Copy of the state: free stack bottom-to-top into free_stack_out (room for
 * num_blocks entries, *free_count_out entries written) and every block's
 * count into refcounts_out (num_blocks entries).  Host buffers. */
pa_status pa_alloc_dump(const pa_allocator* a, int32_t* free_stack_out, int32_t* free_count_out,
                        int32_t* refcounts_out);

/* ------------------------------------------------ prefix cache (host) */

/* Automatic prefix caching ([DEV] section 5, 2 "Automatic Prefix Caching":
 * a request whose tokens match a previously computed sequence gets the
 * matching physical blocks from a hash table mapped into its block table,
 * skipping their prefill; [HI] "Prefix caching: share the system prompt").
 * The pages name no hash or policy; the readings taken:
 *   - only full blocks are cached;
 *   - block j of a token sequence is keyed by FNV-1a-64 over the
 *     little-endian bytes of block j-1's key (0 for block 0) followed by
 *     block j's token ids as 32-bit values (pa_prefix_block_key), so a key
 *     stands for the whole prefix up to its block;
 *   - a hit is verified against the stored parent key and token ids, so a
 *     hash collision never maps a wrong block;
 *   - the cache holds one reference on every cached block;
 *   - eviction releases blocks that only the cache still references, least
 *     recently used first (one match or insert is one use), deeper blocks
 *     first within a use, then by key.
 * Not thread-safe: the caller serialises calls on a cache and its allocator.
 * The allocator must outlive the cache. */
typedef struct pa_prefix_cache pa_prefix_cache;

/* A cache over `alloc` for blocks of `block_size` tokens. */
pa_status pa_prefix_create(pa_allocator* alloc, int32_t block_size, pa_prefix_cache** out);
/* Release the cache's references (in insertion order) and free it. */
void pa_prefix_destroy(pa_prefix_cache* c);
/* Key of a block of `num_tokens` token ids whose previous block has key
 * `parent_key` (0 for the first block).  0 for invalid input. */
uint64_t pa_prefix_block_key(uint64_t parent_key, const int32_t* tokens, int32_t num_tokens);
/* Cached blocks, -1 for a null cache. */
int32_t pa_prefix_size(const pa_prefix_cache* c);
/* Map the longest cached full-block prefix of a request's token ids (host
 * [num_tokens]) into table_row[0 .. *matched_blocks) (host, `capacity`
 * entries); each mapped block gains a reference for the request.  The
 * request's prefill can skip *matched_blocks * block_size tokens. */
pa_status pa_prefix_match(pa_prefix_cache* c, const int32_t* tokens, int32_t num_tokens, int32_t* table_row,
                          int32_t capacity, int32_t* matched_blocks);
/* Cache the full blocks of a computed sequence: tokens (host [num_tokens])
 * whose KV sits in table_row[0 .. num_blocks).  Blocks already cached under
 * their key are only marked used; insertion stops at a key held by other
 * contents or at a block cached under another key.  *inserted = new
 * entries.  PA_ERR_RANGE / PA_ERR_INVALID for an id out of range / free, with
 * nothing changed. */
pa_status pa_prefix_insert(pa_prefix_cache* c, const int32_t* tokens, int32_t num_tokens, const int32_t* table_row,
                           int32_t num_blocks, int32_t* inserted);
/* Release up to `max_blocks` cached blocks that only the cache references
 * (they return to the allocator's pool); *evicted = how many. */
pa_status pa_prefix_evict(pa_prefix_cache* c, int32_t max_blocks, int32_t* evicted);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
