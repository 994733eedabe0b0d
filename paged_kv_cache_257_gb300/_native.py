"""ctypes declarations of ``libpagedattn.so`` (the C ABI in include/pagedattn.h).

Loading fails loudly when the library has not been built: there is no
Python or CPU fallback for any entry point.
"""

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedattn.so")

c_int32, c_int64, c_uint64, c_size_t = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t
c_float, c_void_p, c_char_p = ctypes.c_float, ctypes.c_void_p, ctypes.c_char_p
P_int32, P_int64 = ctypes.POINTER(c_int32), ctypes.POINTER(c_int64)

STATUS = {0: "PA_OK", 1: "PA_ERR_INVALID", 2: "PA_ERR_OOM", 3: "PA_ERR_RANGE", 4: "PA_ERR_UNSUPPORTED",
          5: "PA_ERR_CUDA", 6: "PA_ERR_DEVICE_FLAG"}
DTYPE = {"f32": 0, "f16": 1, "bf16": 2, "fp8_e4m3": 3}

DEVFLAG_SLOT_RANGE = 1
DEVFLAG_BLOCK_RANGE = 2
DEVFLAG_CONTEXT_RANGE = 4
DEVFLAG_TIMEOUT = 8
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024   # PA_NOALLOC_SCRATCH_BYTES
DECODE_KERNEL = {"auto": 0, "cta": 1, "warp": 2}   # PA_DECODE_KERNEL_*


class CacheDescC(ctypes.Structure):
    _fields_ = [("num_blocks", c_int32), ("block_size", c_int32), ("num_kv_heads", c_int32),
                ("head_dim", c_int32), ("kv_dtype", ctypes.c_int), ("k_scale", c_float), ("v_scale", c_float)]


P_desc = ctypes.POINTER(CacheDescC)

# name -> (restype, argtypes)
SIGNATURES = {
    "pa_version": (c_char_p, []),
    "pa_status_string": (c_char_p, [ctypes.c_int]),
    "pa_dtype_size": (c_size_t, [ctypes.c_int]),
    "pa_kv_bytes_per_token": (c_uint64, [c_int32, c_int32, c_int32, ctypes.c_int]),
    "pa_compute_slot_mapping": (ctypes.c_int, [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32,
                                               c_void_p]),
    "pa_kv_append": (ctypes.c_int, [P_desc, c_void_p, c_void_p, ctypes.c_int, c_void_p, c_int32, c_void_p,
                                    c_void_p, c_void_p, c_void_p]),
    "pa_copy_blocks": (ctypes.c_int, [P_desc, c_void_p, c_void_p, c_void_p, c_void_p, c_int32, c_void_p,
                                      c_void_p]),
    "pa_decode_partition_size": (c_int32, [P_desc, c_int32, c_int32, c_int32, c_int32]),
    "pa_decode_plan_partition": (c_int32, [P_desc, c_int32, c_int32, c_int32, c_void_p, c_int32]),
    "pa_decode_workspace_size": (c_size_t, [P_desc, c_int32, c_int32, c_int32, c_int32]),
    "pa_decode_attention": (ctypes.c_int, [P_desc, c_void_p, ctypes.c_int, c_int32, c_void_p, c_void_p, c_void_p,
                                           c_int32, c_void_p, c_int32, c_float, c_int32, c_void_p, c_size_t,
                                           c_void_p, ctypes.c_int, c_void_p, c_void_p]),
    "pa_decode_attention_window": (ctypes.c_int, [P_desc, c_void_p, ctypes.c_int, c_int32, c_void_p, c_void_p,
                                                  c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_float, c_int32,
                                                  c_void_p, c_size_t, c_void_p, ctypes.c_int, c_void_p, c_void_p]),
    "pa_decode_attention_noalloc": (ctypes.c_int, [P_desc, c_void_p, ctypes.c_int, c_int32, c_void_p, c_void_p,
                                                   c_void_p, c_int32, c_void_p, c_int32, c_float, c_int32, c_void_p,
                                                   ctypes.c_int, c_void_p, c_void_p]),
    "pa_read_device_status": (ctypes.c_int, [c_void_p, P_int32, c_int32, c_void_p]),
    "pa_set_decode_deterministic": (None, [c_int32]),
    "pa_get_decode_deterministic": (c_int32, []),
    "pa_set_decode_kernel": (ctypes.c_int, [c_int32]),
    "pa_get_decode_kernel": (c_int32, []),
    "pa_alloc_create": (ctypes.c_int, [c_int32, c_uint64, ctypes.POINTER(c_void_p)]),
    "pa_alloc_destroy": (None, [c_void_p]),
    "pa_alloc_num_blocks": (c_int32, [c_void_p]),
    "pa_alloc_free_count": (c_int32, [c_void_p]),
    "pa_alloc_refcount": (c_int32, [c_void_p, c_int32]),
    "pa_alloc_block": (ctypes.c_int, [c_void_p, P_int32]),
    "pa_alloc_incref": (ctypes.c_int, [c_void_p, c_int32]),
    "pa_alloc_decref": (ctypes.c_int, [c_void_p, c_int32]),
    "pa_alloc_cow": (ctypes.c_int, [c_void_p, c_int32, P_int32, P_int32]),
    "pa_alloc_append_slot": (ctypes.c_int, [c_void_p, c_void_p, c_int32, P_int32, c_int32, c_int32, P_int64,
                                            P_int32, P_int32]),
    "pa_alloc_fork": (ctypes.c_int, [c_void_p, c_void_p, c_int32]),
    "pa_alloc_free_sequence": (ctypes.c_int, [c_void_p, c_void_p, c_int32]),
    "pa_prefix_create": (ctypes.c_int, [c_void_p, c_int32, c_void_p]),
    "pa_prefix_destroy": (None, [c_void_p]),
    "pa_prefix_block_key": (c_uint64, [c_uint64, c_void_p, c_int32]),
    "pa_prefix_size": (c_int32, [c_void_p]),
    "pa_prefix_match": (ctypes.c_int, [c_void_p, c_void_p, c_int32, c_void_p, c_int32, P_int32]),
    "pa_prefix_insert": (ctypes.c_int, [c_void_p, c_void_p, c_int32, c_void_p, c_int32, P_int32]),
    "pa_prefix_evict": (ctypes.c_int, [c_void_p, c_int32, P_int32]),
    "pa_alloc_truncate": (ctypes.c_int, [c_void_p, c_void_p, c_int32, P_int32, P_int32, P_int32, c_int32, c_int32]),
    "pa_alloc_dump": (ctypes.c_int, [c_void_p, c_void_p, P_int32, c_void_p]),
}

_lock = threading.Lock()
_lib = None


class NativeError(RuntimeError):
    """A library call returned a status other than PA_OK."""

    def __init__(self, fn, status):
        self.status = STATUS.get(status, f"status {status}")
        super().__init__(f"{fn} failed: {self.status}")


def load(path):
    """A built copy of the library at ``path`` with every call's signature set."""
    L = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    """The loaded library (built beforehand by ``paged_kv_cache_257_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it first with "
                                   "paged_kv_cache_257_gb300.build.build() (nvcc, sm_103a); "
                                   "there is no fallback implementation")
            _lib = load(LIB_PATH)
    return _lib


def check(fn_name, status):
    if status != 0:
        raise NativeError(fn_name, status)
