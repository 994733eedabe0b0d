// Decode attention that allocates nothing, for callers that cannot call
// cudaMalloc: code running inside a host framework or server that owns all
// device memory through its own allocator and forbids other allocations,
// decode loops that must not stall every stream on the implicit device
// synchronisation of cudaMalloc, and deployments whose device memory
// footprint is fixed up front.  The caller still passes every input and
// output buffer; only the split-context workspace comes from a fixed array
// in device memory that this library owns.
#include <mutex>
#include <vector>

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode.h"
#include "pagedattn.h"

namespace {

// The workspace of pa_decode_attention_noalloc.  Every GPU that loads the
// library holds one copy of this array until the process exits.
static_assert(PA_NOALLOC_SCRATCH_BYTES % 256 == 0, "scratch size must keep 256-byte alignment");
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

// The array's device address belongs to one CUDA context: after a
// cudaDeviceReset the device's next context holds the array elsewhere.
// Each device's entry records the context it was looked up in (its driver
// id), so a new context is noticed and the address asked for again.
struct ScratchEntry {
    unsigned long long ctx_id = 0;
    void* ptr = nullptr;
};

std::mutex g_mutex;
std::vector<ScratchEntry> g_scratch;   // per device

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Driver id of the calling thread's current context (0 if none answers).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
        get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

// Device address of the array on the current device.  In host code the
// array's name stands for a host-side shadow, never the device memory, so
// the address is asked of the runtime with the device current, once per
// device and context, and cached; the array is zero-filled then.
pa_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    unsigned long long ctx = current_context_id();
    if (ctx == 0) {   // no context current in this thread yet: the runtime makes the device's current
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return PA_ERR_CUDA;
        ctx = current_context_id();
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (dev >= static_cast<int>(g_scratch.size())) g_scratch.resize(dev + 1);
    ScratchEntry& e = g_scratch[dev];
    if (e.ptr == nullptr || e.ctx_id != ctx) {
        e.ptr = nullptr;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        if (cudaMemset(p, 0, PA_NOALLOC_SCRATCH_BYTES) != cudaSuccess) return PA_ERR_CUDA;
        if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
        e.ptr = p;
        e.ctx_id = ctx;
    }
    *out = e.ptr;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_attention_noalloc(const pa_cache_desc* cache, const void* q, pa_dtype q_dtype,
                                                 int32_t num_q_heads, const void* k_cache, const void* v_cache,
                                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                                 const int32_t* context_lens, int32_t batch, float scale,
                                                 int32_t partition_size, void* out, pa_dtype out_dtype,
                                                 int32_t* device_status, void* stream) {
    const size_t need = pa_decode_workspace_size(cache, batch, num_q_heads, max_blocks_per_seq, partition_size);
    if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_RANGE;
    void* ws = nullptr;
    if (need > 0) {
        if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PA_ERR_INVALID;
        pa_status st = scratch_address(&ws);
        if (st != PA_OK) return st;
        // The array keeps the previous call's contents.  Its front holds the
        // counters a call expects at zero (the merge tickets):
        // clear them on the caller's stream, ahead of the kernels.
        const size_t counters =
            pa::decode_counter_bytes(cache, batch, num_q_heads, max_blocks_per_seq, partition_size);
        if (cudaMemsetAsync(ws, 0, counters, static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    }
    return pa_decode_attention(cache, q, q_dtype, num_q_heads, k_cache, v_cache, block_tables, max_blocks_per_seq,
                               context_lens, batch, scale, partition_size, ws, need, out, out_dtype, device_status,
                               stream);
}
