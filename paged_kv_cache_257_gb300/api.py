"""Thin Python binding over the C ABI: argument marshalling only.

Every step of the hot path runs in the library's CUDA kernels; torch is used
here for device memory (tensors the library reads and writes) and for the
current CUDA stream.  Names follow the C ABI (``pa_kv_append`` ->
``kv_append`` and so on).
"""

import ctypes
import dataclasses

import numpy as np
import torch

from . import _native
from ._native import DTYPE, NativeError, check, lib

TORCH_STORAGE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16, "fp8_e4m3": torch.uint8}
_FROM_TORCH = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


@dataclasses.dataclass
class CacheDesc:
    """One layer's paged KV cache: pools ``[num_blocks, num_kv_heads, block_size, head_dim]``."""

    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_dim: int
    kv_dtype: str = "bf16"
    k_scale: float = 1.0
    v_scale: float = 1.0

    def c(self):
        """The C struct (built once per distinct field values: calls are on the hot path)."""
        key = (self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim, self.kv_dtype, self.k_scale,
               self.v_scale)
        if self.__dict__.get("_c_key") != key:
            self.__dict__["_c"] = _native.CacheDescC(self.num_blocks, self.block_size, self.num_kv_heads,
                                                     self.head_dim, DTYPE[self.kv_dtype], self.k_scale, self.v_scale)
            self.__dict__["_c_key"] = key
        return self.__dict__["_c"]

    @property
    def pool_shape(self):
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    def new_pools(self, device="cuda", fill=None):
        """Allocate the K and V pools (torch, device memory); optionally fill raw bytes."""
        k = torch.empty(self.pool_shape, dtype=TORCH_STORAGE[self.kv_dtype], device=device)
        v = torch.empty_like(k)
        if fill is not None:
            k.view(torch.uint8).fill_(fill)
            v.view(torch.uint8).fill_(fill)
        return k, v


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_of(t, what):
    if t.dtype not in _FROM_TORCH:
        raise TypeError(f"{what}: unsupported dtype {t.dtype}")
    return _FROM_TORCH[t.dtype]


def _need(t, what, dtype=None, cuda=True):
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if cuda and not t.is_cuda:
        raise ValueError(f"{what} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")


# ------------------------------------------------------------------ info

def version():
    return lib().pa_version().decode()


def dtype_size(dtype):
    return int(lib().pa_dtype_size(DTYPE[dtype]))


def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, dtype):
    return int(lib().pa_kv_bytes_per_token(n_layers, n_kv_heads, head_dim, DTYPE[dtype]))


def compute_slot_mapping(block_tables, seq_ids, positions, block_size):
    """int64 slots of (sequence, position) pairs from host block tables (numpy)."""
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sid = np.ascontiguousarray(seq_ids, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    out = np.empty(len(sid), dtype=np.int64)
    st = lib().pa_compute_slot_mapping(bt.ctypes.data, bt.shape[0], bt.shape[1], block_size, sid.ctypes.data,
                                      pos.ctypes.data, len(sid), out.ctypes.data)
    check("pa_compute_slot_mapping", st)
    return out


# ---------------------------------------------------------- device calls

def kv_append(desc, k, v, slot_mapping, k_cache, v_cache, status=None, stream=None):
    """Write new tokens' K/V rows ``[T, Hkv, D]`` into their slots (``pa_kv_append``)."""
    for t, n in ((k, "k"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, n)
    _need(slot_mapping, "slot_mapping", torch.int64)
    src = _dtype_of(k, "k")
    if v.dtype != k.dtype:
        raise TypeError("k and v must share a dtype")
    c = desc.c()
    st = lib().pa_kv_append(ctypes.byref(c), _ptr(k), _ptr(v), DTYPE[src], _ptr(slot_mapping),
                            slot_mapping.numel(), _ptr(k_cache), _ptr(v_cache), _ptr(status), _stream(stream))
    check("pa_kv_append", st)


def copy_blocks(desc, k_cache, v_cache, src_blocks, dst_blocks, status=None, stream=None):
    """Copy whole physical blocks src -> dst in both pools (``pa_copy_blocks``)."""
    _need(src_blocks, "src_blocks", torch.int32)
    _need(dst_blocks, "dst_blocks", torch.int32)
    c = desc.c()
    st = lib().pa_copy_blocks(ctypes.byref(c), _ptr(k_cache), _ptr(v_cache), _ptr(src_blocks), _ptr(dst_blocks),
                              src_blocks.numel(), _ptr(status), _stream(stream))
    check("pa_copy_blocks", st)


def partition_size(desc, batch, num_q_heads, max_blocks_per_seq, requested=0):
    c = desc.c()
    return int(lib().pa_decode_partition_size(ctypes.byref(c), batch, num_q_heads, max_blocks_per_seq, requested))


def plan_partition(desc, batch, num_q_heads, max_blocks_per_seq, context_lens=None, num_sms=0):
    """Partition size for a batch whose context lengths are known on the host
    (``context_lens``: host int sequence, or None for every sequence full);
    ``num_sms`` <= 0 asks the current device."""
    c = desc.c()
    arr = None
    if context_lens is not None:
        arr = np.ascontiguousarray(np.asarray(context_lens), dtype=np.int32)
        if arr.shape != (batch,):
            raise ValueError(f"context_lens must hold {batch} lengths, got shape {arr.shape}")
    p = int(lib().pa_decode_plan_partition(ctypes.byref(c), batch, num_q_heads, max_blocks_per_seq,
                                           None if arr is None else arr.ctypes.data, num_sms))
    if p <= 0:
        raise ValueError("pa_decode_plan_partition rejected its arguments")
    return p


def decode_workspace_size(desc, batch, num_q_heads, max_blocks_per_seq, partition=0):
    c = desc.c()
    return int(lib().pa_decode_workspace_size(ctypes.byref(c), batch, num_q_heads, max_blocks_per_seq, partition))


def decode_attention(desc, q, k_cache, v_cache, block_tables, context_lens, scale, partition=0, workspace=None,
                     out=None, out_dtype=None, status=None, stream=None, context_starts=None):
    """Single-query paged decode attention (``pa_decode_attention``); returns ``out``.

    ``q`` is ``[batch, num_q_heads, head_dim]``; ``block_tables`` int32
    ``[batch, max_blocks]``; ``context_lens`` int32 ``[batch]``.  ``out`` and
    the split-context ``workspace`` are allocated with torch when not given; a
    given workspace is passed with its size, which the library checks.
    ``context_starts`` (device int32 ``[batch]``) restricts each sequence to
    the positions from its start on (``pa_decode_attention_window``).
    """
    _need(q, "q")
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    if context_starts is not None:
        _need(context_starts, "context_starts", torch.int32)
        if context_starts.shape != context_lens.shape:
            raise ValueError("context_starts must have the shape of context_lens")
    batch, hq, d = q.shape
    max_blocks = block_tables.shape[1]
    if out is None:
        od = out_dtype or "f32"
        out = torch.empty((batch, hq, d), dtype=TORCH_STORAGE[od], device=q.device)
    _need(out, "out")
    od = _dtype_of(out, "out")
    if workspace is None:
        need = decode_workspace_size(desc, batch, hq, max_blocks, partition)
        workspace = new_workspace(need, q.device) if need else None
    need = workspace.numel() * workspace.element_size() if workspace is not None else 0
    c = desc.c()
    if context_starts is None:
        st = lib().pa_decode_attention(ctypes.byref(c), _ptr(q), DTYPE[_dtype_of(q, "q")], hq, _ptr(k_cache),
                                       _ptr(v_cache), _ptr(block_tables), max_blocks, _ptr(context_lens), batch,
                                       float(scale), partition, _ptr(workspace) if need else None,
                                       need if need else 0, _ptr(out), DTYPE[od], _ptr(status), _stream(stream))
        check("pa_decode_attention", st)
    else:
        st = lib().pa_decode_attention_window(ctypes.byref(c), _ptr(q), DTYPE[_dtype_of(q, "q")], hq,
                                              _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks,
                                              _ptr(context_lens), _ptr(context_starts), batch, float(scale),
                                              partition, _ptr(workspace) if need else None, need if need else 0,
                                              _ptr(out), DTYPE[od], _ptr(status), _stream(stream))
        check("pa_decode_attention_window", st)
    return out


def decode_attention_noalloc(desc, q, k_cache, v_cache, block_tables, context_lens, scale, out, partition=0,
                             status=None, stream=None):
    """``pa_decode_attention_noalloc``: decode attention with the library's static workspace.

    For callers that must not allocate device memory: the library's own array
    of 8 MiB per GPU replaces the workspace, and this wrapper allocates
    nothing either, so ``out`` ([batch, num_q_heads, head_dim], f32 / f16 /
    bf16) is required.  Raises NativeError("PA_ERR_RANGE") when the
    problem's workspace does not fit the array.
    """
    _need(q, "q")
    _need(block_tables, "block_tables", torch.int32)
    _need(context_lens, "context_lens", torch.int32)
    if out is None:
        raise ValueError("decode_attention_noalloc allocates nothing: pass the output tensor as out")
    batch, hq, d = q.shape
    _need(out, "out")
    c = desc.c()
    st = lib().pa_decode_attention_noalloc(ctypes.byref(c), _ptr(q), DTYPE[_dtype_of(q, "q")], hq, _ptr(k_cache),
                                           _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
                                           _ptr(context_lens), batch, float(scale), partition, _ptr(out),
                                           DTYPE[_dtype_of(out, "out")], _ptr(status), _stream(stream))
    check("pa_decode_attention_noalloc", st)
    return out


def set_decode_deterministic(on):
    """``pa_set_decode_deterministic``: True gives bit-reproducible decode
    results (every chunk on a fixed warp); False (the default) lets the
    warps of a CTA share out an item's last chunks, which is faster and
    reproducible to bf16 rounding of the probabilities only.  Process-wide;
    returns the previous setting."""
    prev = bool(lib().pa_get_decode_deterministic())
    lib().pa_set_decode_deterministic(1 if on else 0)
    return prev


def decode_deterministic():
    """The current ``pa_set_decode_deterministic`` setting."""
    return bool(lib().pa_get_decode_deterministic())


def set_decode_kernel(kernel):
    """``pa_set_decode_kernel``: "auto" (the library picks per call), "cta"
    (a CTA of four warps per work item) or "warp" (one warp per work item)
    for every later tensor-core decode call of the process.  Returns the
    previous setting."""
    from ._native import DECODE_KERNEL
    names = {v: k for k, v in DECODE_KERNEL.items()}
    prev = names[int(lib().pa_get_decode_kernel())]
    check("pa_set_decode_kernel", lib().pa_set_decode_kernel(DECODE_KERNEL[kernel]))
    return prev


def decode_kernel():
    """The current ``pa_set_decode_kernel`` setting."""
    from ._native import DECODE_KERNEL
    return {v: k for k, v in DECODE_KERNEL.items()}[int(lib().pa_get_decode_kernel())]


def new_workspace(nbytes, device="cuda"):
    """A zero-filled decode workspace (the library keeps its counters zero between calls)."""
    return torch.zeros(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def new_status(device="cuda"):
    """A zeroed device status word for the ``status=`` arguments."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def read_device_status(status, reset=True, stream=None):
    """Flags raised on the device since the word was last cleared (synchronises the stream)."""
    flags = ctypes.c_int32(0)
    st = lib().pa_read_device_status(_ptr(status), ctypes.byref(flags), 1 if reset else 0, _stream(stream))
    if st not in (0, 6):
        check("pa_read_device_status", st)
    return int(flags.value)


# ------------------------------------------------------------- allocator

_ALLOC_STATUS = {2: "OOM", 1: "INVALID", 3: "RANGE"}


class AllocError(Exception):
    """Allocator failure; ``status`` is "OOM", "INVALID" or "RANGE"."""

    def __init__(self, status, fn):
        super().__init__(f"{fn}: {status}")
        self.status = status


def _alloc_check(fn, st):
    if st != 0:
        if st in _ALLOC_STATUS:
            raise AllocError(_ALLOC_STATUS[st], fn)
        check(fn, st)


class BlockAllocator:
    """The library's host block allocator (``pa_alloc_*``), same methods as the model."""

    def __init__(self, num_blocks, seed=0):
        h = ctypes.c_void_p()
        _alloc_check("pa_alloc_create", lib().pa_alloc_create(num_blocks, seed, ctypes.byref(h)))
        self._h = h
        self.num_blocks = num_blocks

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib().pa_alloc_destroy(h)
            self._h = None

    def alloc(self):
        b = ctypes.c_int32()
        _alloc_check("pa_alloc_block", lib().pa_alloc_block(self._h, ctypes.byref(b)))
        return b.value

    def incref(self, b):
        _alloc_check("pa_alloc_incref", lib().pa_alloc_incref(self._h, b))

    def decref(self, b):
        _alloc_check("pa_alloc_decref", lib().pa_alloc_decref(self._h, b))

    def cow(self, b):
        nb, copied = ctypes.c_int32(), ctypes.c_int32()
        _alloc_check("pa_alloc_cow", lib().pa_alloc_cow(self._h, b, ctypes.byref(nb), ctypes.byref(copied)))
        return nb.value, bool(copied.value)

    def append_slot(self, table_row, num_blocks, position, block_size):
        """Slot for logical token ``position``; updates ``table_row`` (a list) in place.

        Returns ``(slot, num_blocks, cow)`` with ``cow`` = ``(src, dst)`` or None."""
        arr = (ctypes.c_int32 * len(table_row))(*table_row)
        n = ctypes.c_int32(num_blocks)
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        st = lib().pa_alloc_append_slot(self._h, arr, len(table_row), ctypes.byref(n), position, block_size,
                                        ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst))
        _alloc_check("pa_alloc_append_slot", st)
        table_row[:] = list(arr)
        return slot.value, n.value, (None if src.value < 0 else (src.value, dst.value))

    def fork(self, table_row, num_blocks):
        arr = np.ascontiguousarray(table_row[:num_blocks], dtype=np.int32)
        _alloc_check("pa_alloc_fork", lib().pa_alloc_fork(self._h, arr.ctypes.data, num_blocks))

    def free_sequence(self, table_row, num_blocks):
        arr = np.ascontiguousarray(table_row[:num_blocks], dtype=np.int32)
        _alloc_check("pa_alloc_free_sequence", lib().pa_alloc_free_sequence(self._h, arr.ctypes.data, num_blocks))

    def truncate(self, table_row, num_blocks, start, length, keep, block_size):
        """Keep the last ``keep`` tokens of a sequence (``pa_alloc_truncate``);
        updates ``table_row`` (a list) in place and returns ``(num_blocks,
        start, length)``."""
        arr = (ctypes.c_int32 * len(table_row))(*table_row)
        n, s0, ln = ctypes.c_int32(num_blocks), ctypes.c_int32(start), ctypes.c_int32(length)
        st = lib().pa_alloc_truncate(self._h, arr, len(table_row), ctypes.byref(n), ctypes.byref(s0),
                                     ctypes.byref(ln), keep, block_size)
        _alloc_check("pa_alloc_truncate", st)
        table_row[:] = list(arr)
        return n.value, s0.value, ln.value

    @property
    def free_count(self):
        return int(lib().pa_alloc_free_count(self._h))

    def refcount(self, b):
        return int(lib().pa_alloc_refcount(self._h, b))

    @property
    def ref(self):
        return self.dump()[1]

    def dump(self):
        free = np.empty(self.num_blocks, dtype=np.int32)
        ref = np.empty(self.num_blocks, dtype=np.int32)
        nf = ctypes.c_int32()
        _alloc_check("pa_alloc_dump", lib().pa_alloc_dump(self._h, free.ctypes.data, ctypes.byref(nf),
                                                           ref.ctypes.data))
        return [int(x) for x in free[:nf.value]], [int(x) for x in ref]


__all__ = ["CacheDesc", "BlockAllocator", "AllocError", "NativeError", "version", "dtype_size",
           "kv_bytes_per_token", "compute_slot_mapping", "kv_append", "copy_blocks", "partition_size", "plan_partition",
           "PrefixCache",
           "decode_workspace_size", "decode_attention", "decode_attention_noalloc", "set_decode_kernel", "decode_kernel", "new_status", "new_workspace", "read_device_status"]


class PrefixCache:
    """The library's prefix cache (``pa_prefix_*``) over a ``BlockAllocator``;
    same methods as the oracle's model.  Holds its allocator alive."""

    def __init__(self, allocator, block_size):
        h = ctypes.c_void_p()
        _alloc_check("pa_prefix_create", lib().pa_prefix_create(allocator._h, block_size, ctypes.byref(h)))
        self._h, self._alloc, self.bs = h, allocator, block_size

    def __del__(self):
        self.destroy()

    def destroy(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            lib().pa_prefix_destroy(h)
        self._h = None

    @staticmethod
    def block_key(parent_key, tokens):
        arr = np.ascontiguousarray(tokens, dtype=np.int32)
        return int(lib().pa_prefix_block_key(parent_key, arr.ctypes.data, arr.size))

    @property
    def size(self):
        return int(lib().pa_prefix_size(self._h))

    def match(self, tokens, table_row):
        """Maps the cached prefix into ``table_row`` (a list, updated in place); returns the blocks matched."""
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        arr = (ctypes.c_int32 * len(table_row))(*table_row)
        m = ctypes.c_int32()
        _alloc_check("pa_prefix_match", lib().pa_prefix_match(self._h, toks.ctypes.data, toks.size, arr,
                                                               len(table_row), ctypes.byref(m)))
        table_row[:] = list(arr)
        return m.value

    def insert(self, tokens, table_row, num_blocks):
        toks = np.ascontiguousarray(tokens, dtype=np.int32)
        row = np.ascontiguousarray(table_row[:num_blocks], dtype=np.int32)
        made = ctypes.c_int32()
        _alloc_check("pa_prefix_insert", lib().pa_prefix_insert(self._h, toks.ctypes.data, toks.size,
                                                                 row.ctypes.data, num_blocks, ctypes.byref(made)))
        return made.value

    def evict(self, max_blocks):
        n = ctypes.c_int32()
        _alloc_check("pa_prefix_evict", lib().pa_prefix_evict(self._h, max_blocks, ctypes.byref(n)))
        return n.value
