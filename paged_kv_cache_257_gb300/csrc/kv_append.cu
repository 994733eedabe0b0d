// KV append (slot scatter with optional FP8 quantisation) and whole-block copy.
//
// dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
// PagedAttention Fixes It", section 1 "Why Transformers Need a KV Cache": each
// decode step computes the new token's K and V and appends them to the
// cache; section 4 "How the Architecture Works": the token goes into the
// slot of the physical block its block table names; section 6 item 4 and
// hyperinfer.ai "KV quantization cuts memory in half": the cache may hold
// one-byte FP8 values.  Section 5 "Zero-Copy Forking": a write into a shared
// block first copies it (pa_copy_blocks).
//
// One thread moves a pack of 8 consecutive elements of one (token, KV head)
// row: 16-byte loads and stores for 16-bit types, 32-byte float32 sources,
// 8-byte FP8 destinations.  The work is tiny and launch-bound; the grid is
// sized to the work, capped at a few waves of the GPU.
#include <algorithm>

#include "common.cuh"
#include "decode.h"

namespace pa {
namespace {

constexpr int kPack = 8;
constexpr int kAppendThreads = 256;

template <pa_dtype SRC>
__device__ __forceinline__ void load_pack_f32(const void* base, int64_t elem, float (&x)[kPack]) {
    if constexpr (SRC == PA_F32) {
        const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
        float4 a = __ldg(p), b = __ldg(p + 1);
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
        using T = typename Elem<SRC>::type;
        uint4 raw = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(base) + elem));
        const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
        for (int i = 0; i < kPack; ++i) x[i] = to_float<SRC>(e, i);
    }
}

// One pack in registers, already in the cache's type: load() reads (and
// converts) the source, store() writes the slot; split so that the source
// read need not wait for the slot.
template <pa_dtype SRC, pa_dtype DST>
struct Pack {
    static constexpr int kWords = kPack * Elem<DST>::bytes / 4;
    alignas(16) uint32_t w[kWords];

    __device__ __forceinline__ void load(const void* src, int64_t src_elem, float scale) {
        if constexpr (SRC == DST) {
            using T = typename Elem<DST>::type;
            const uint4* s = reinterpret_cast<const uint4*>(static_cast<const T*>(src) + src_elem);
#pragma unroll
            for (int i = 0; i < kWords / 4; ++i) reinterpret_cast<uint4*>(w)[i] = __ldg(s + i);
        } else if constexpr (DST == PA_FP8_E4M3) {
            float x[kPack];
            load_pack_f32<SRC>(src, src_elem, x);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint32_t lo = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(x[4 * i + 0], scale), __fdiv_rn(x[4 * i + 1], scale)), __NV_SATFINITE,
                    __NV_E4M3);
                uint32_t hi = __nv_cvt_float2_to_fp8x2(
                    make_float2(__fdiv_rn(x[4 * i + 2], scale), __fdiv_rn(x[4 * i + 3], scale)), __NV_SATFINITE,
                    __NV_E4M3);
                w[i] = (lo & 0xFFFFu) | (hi << 16);
            }
        } else {
            static_assert(SRC == PA_F32, "only float32 sources narrow to 16-bit caches");
            float x[kPack];
            load_pack_f32<SRC>(src, src_elem, x);
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = pack2<DST == PA_BF16>(x[2 * i], x[2 * i + 1]);
        }
    }

    __device__ __forceinline__ void store(void* dst, int64_t dst_elem) const {
        uint8_t* d = static_cast<uint8_t*>(dst) + dst_elem * Elem<DST>::bytes;
        if constexpr (kWords == 2) {
            *reinterpret_cast<uint2*>(d) = make_uint2(w[0], w[1]);
        } else {
#pragma unroll
            for (int i = 0; i < kWords / 4; ++i) reinterpret_cast<uint4*>(d)[i] = reinterpret_cast<const uint4*>(w)[i];
        }
    }
};

template <pa_dtype SRC, pa_dtype DST>
__global__ void __launch_bounds__(kAppendThreads)
kv_append_kernel(const void* __restrict__ k, const void* __restrict__ v, const int64_t* __restrict__ slots,
                 int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                 int64_t num_slots, void* __restrict__ k_cache, void* __restrict__ v_cache, float k_scale,
                 float v_scale, int32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int64_t packs_per_row = head_dim / kPack;
    const int64_t per_tensor = static_cast<int64_t>(num_tokens) * num_kv_heads * packs_per_row;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t p = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; p < 2 * per_tensor;
         p += stride) {
        const bool is_v = p >= per_tensor;
        const int64_t r = is_v ? p - per_tensor : p;
        const int64_t row = r / packs_per_row;           // token * num_kv_heads + head
        const int64_t chunk = r - row * packs_per_row;
        const int64_t t = row / num_kv_heads;
        const int64_t h = row - t * num_kv_heads;
        const int64_t slot = __ldg(slots + t);
        Pack<SRC, DST> pk;
        pk.load(is_v ? v : k, row * head_dim + chunk * kPack, is_v ? v_scale : k_scale);
        if (slot < 0 || slot >= num_slots) {
            if (!is_v && h == 0 && chunk == 0) raise_flag(status, PA_DEVFLAG_SLOT_RANGE);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        pk.store(is_v ? v_cache : k_cache, ((blk * num_kv_heads + h) * block_size + off) * head_dim + chunk * kPack);
    }
}

__global__ void __launch_bounds__(kAppendThreads)
copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache, const int32_t* __restrict__ src,
                   const int32_t* __restrict__ dst, int32_t num_blocks, int64_t block_vec16,
                   int32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int32_t pair = blockIdx.y;
    const int32_t s = __ldg(src + pair), d = __ldg(dst + pair);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (blockIdx.x == 0 && blockIdx.z == 0 && threadIdx.x == 0) raise_flag(status, PA_DEVFLAG_BLOCK_RANGE);
        return;
    }
    uint4* pool = blockIdx.z == 0 ? k_cache : v_cache;
    const uint4* from = pool + static_cast<int64_t>(s) * block_vec16;
    uint4* to = pool + static_cast<int64_t>(d) * block_vec16;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < block_vec16;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        to[i] = from[i];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Host check shared by the entry points: a well-formed cache descriptor.
pa_status check_cache_desc(const pa_cache_desc* c) {
    if (c == nullptr) return PA_ERR_INVALID;
    if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
        return PA_ERR_INVALID;
    if (c->block_size != 8 && c->block_size != 16 && c->block_size != 32) return PA_ERR_UNSUPPORTED;
    if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (c->kv_dtype != PA_F32 && c->kv_dtype != PA_F16 && c->kv_dtype != PA_BF16 && c->kv_dtype != PA_FP8_E4M3)
        return PA_ERR_INVALID;
    if (c->kv_dtype == PA_FP8_E4M3) {
        if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f) || !isfinite(c->k_scale) || !isfinite(c->v_scale))
            return PA_ERR_INVALID;
    }
    // slots and tensor-map rows stay well inside int32 / int64 arithmetic
    const int64_t rows = (static_cast<int64_t>(c->num_blocks) + 1) * c->num_kv_heads * c->block_size;
    if (rows >= (int64_t{1} << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

}  // namespace pa

using namespace pa;

namespace {

template <pa_dtype SRC, pa_dtype DST>
cudaError_t launch_append(const pa_cache_desc* c, const void* k, const void* v, const int64_t* slots, int32_t n,
                   void* kc, void* vc, int32_t* status, cudaStream_t stream) {
    const int64_t total = 2ll * n * c->num_kv_heads * (c->head_dim / kPack);
    const int64_t want = (total + kAppendThreads - 1) / kAppendThreads;
    const int blocks = static_cast<int>(std::min<int64_t>(want, 16ll * sm_count()));
    const float ks = DST == PA_FP8_E4M3 ? c->k_scale : 1.f;
    const float vs = DST == PA_FP8_E4M3 ? c->v_scale : 1.f;
    return launch_pdl(kv_append_kernel<SRC, DST>, dim3(blocks), dim3(kAppendThreads), 0, stream, k, v, slots, n,
                      c->num_kv_heads, c->head_dim, c->block_size,
                      static_cast<int64_t>(c->num_blocks) * c->block_size, kc, vc, ks, vs, status);
}

}  // namespace

extern "C" pa_status pa_kv_append(const pa_cache_desc* cache, const void* k, const void* v, pa_dtype src_dtype,
                                  const int64_t* slot_mapping, int32_t num_tokens, void* k_cache,
                                  void* v_cache, int32_t* device_status, void* stream_) {
    pa_status st = check_cache_desc(cache);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(slot_mapping) & 7u) || (reinterpret_cast<uintptr_t>(device_status) & 3u))
        return PA_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    const pa_dtype dst = cache->kv_dtype;
    cudaError_t e;
#define PA_APPEND(SRC_, DST_) e = launch_append<SRC_, DST_>(cache, k, v, slot_mapping, num_tokens, k_cache, v_cache, device_status, s)
    if (dst == PA_F32 && src_dtype == PA_F32) PA_APPEND(PA_F32, PA_F32);
    else if (dst == PA_F16 && src_dtype == PA_F16) PA_APPEND(PA_F16, PA_F16);
    else if (dst == PA_BF16 && src_dtype == PA_BF16) PA_APPEND(PA_BF16, PA_BF16);
    else if (dst == PA_F16 && src_dtype == PA_F32) PA_APPEND(PA_F32, PA_F16);
    else if (dst == PA_BF16 && src_dtype == PA_F32) PA_APPEND(PA_F32, PA_BF16);
    else if (dst == PA_FP8_E4M3 && src_dtype == PA_F32) PA_APPEND(PA_F32, PA_FP8_E4M3);
    else if (dst == PA_FP8_E4M3 && src_dtype == PA_F16) PA_APPEND(PA_F16, PA_FP8_E4M3);
    else if (dst == PA_FP8_E4M3 && src_dtype == PA_BF16) PA_APPEND(PA_BF16, PA_FP8_E4M3);
    else return PA_ERR_UNSUPPORTED;
#undef PA_APPEND
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_copy_blocks(const pa_cache_desc* cache, void* k_cache, void* v_cache,
                                    const int32_t* src_blocks, const int32_t* dst_blocks, int32_t num_pairs,
                                    int32_t* device_status, void* stream_) {
    pa_status st = check_cache_desc(cache);
    if (st != PA_OK) return st;
    if (num_pairs < 0 || num_pairs > 65535) return PA_ERR_INVALID;
    if (num_pairs == 0) return PA_OK;
    if (!k_cache || !v_cache || !src_blocks || !dst_blocks) return PA_ERR_INVALID;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID;
    const int64_t block_bytes = static_cast<int64_t>(cache->num_kv_heads) * cache->block_size * cache->head_dim *
                                static_cast<int64_t>(pa_dtype_size(cache->kv_dtype));
    const int64_t vec = block_bytes / 16;
    const int gx = static_cast<int>(std::min<int64_t>((vec + kAppendThreads - 1) / kAppendThreads, 64));
    dim3 grid(gx, num_pairs, 2);
    cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(kAppendThreads), 0, static_cast<cudaStream_t>(stream_),
                               static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), src_blocks, dst_blocks,
                               cache->num_blocks, vec, device_status);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

extern "C" pa_status pa_read_device_status(int32_t* device_status, int32_t* flags_out, int32_t reset,
                                           void* stream_) {
    if (device_status == nullptr) return PA_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream_);
    int32_t host = 0;
    if (cudaMemcpyAsync(&host, device_status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return PA_ERR_CUDA;
    if (reset && cudaMemsetAsync(device_status, 0, sizeof(int32_t), s) != cudaSuccess) return PA_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
    if (flags_out) *flags_out = host;
    return host ? PA_ERR_DEVICE_FLAG : PA_OK;
}
