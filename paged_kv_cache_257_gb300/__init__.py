"""GB300 paged decode attention: KV append, decode attention, block allocator.

The compute path is ``libpagedattn.so`` (hand-written CUDA for sm_103a behind
a C ABI, declared in ``include/pagedattn.h``); this package is its Python
binding.  Build the library with ``paged_kv_cache_257_gb300.build.build()``.
"""

from .api import (AllocError, BlockAllocator, CacheDesc, NativeError, PrefixCache, compute_slot_mapping, copy_blocks,
                  decode_attention, decode_attention_noalloc, decode_workspace_size, dtype_size, kv_append, kv_bytes_per_token, new_status,
                  new_workspace, partition_size, plan_partition, read_device_status, set_decode_deterministic,
                  decode_deterministic, set_decode_kernel, decode_kernel, version)

__all__ = ["AllocError", "BlockAllocator", "CacheDesc", "NativeError", "PrefixCache", "compute_slot_mapping", "copy_blocks",
           "decode_attention", "decode_attention_noalloc", "decode_workspace_size", "dtype_size", "kv_append", "kv_bytes_per_token",
           "new_status", "new_workspace", "partition_size", "plan_partition", "read_device_status",
           "set_decode_deterministic", "decode_deterministic", "set_decode_kernel", "decode_kernel", "version"]
