"""Paged KV pool model: slot mapping, KV append and the logical gather.

Test infrastructure only (see ``oracle/__init__.py``).

Pool layout (our reading; the pages do not fix one): each of the K and V
pools is an array ``[num_blocks, n_kv_heads, block_size, head_dim]`` of the
cache element type, so the tokens of one (physical block, KV head) pair are
one contiguous run.  A token slot is ``physical_block * block_size + offset``.
"""

import numpy as np

from . import numerics


def new_pool(num_blocks, n_kv_heads, block_size, head_dim, dtype, fill=0):
    """A zeroed (or ``fill``-ed raw storage) pool of the given cache type."""
    shape = (num_blocks, n_kv_heads, block_size, head_dim)
    return np.full(shape, fill, dtype=numerics.STORAGE[dtype])


def slot_of(block_table_row, position, block_size):
    """Slot holding logical token ``position`` of a sequence.

    [DEV] section 4 "How the Architecture Works": the block table maps each
    logical block (``position // block_size``) to the physical block where it
    resides; the token sits at offset ``position % block_size`` inside it
    ([VK] "A minimal PyTorch sketch" takes the in-page offset the same way).
    """
    if position < 0:
        raise ValueError("negative position")
    j = position // block_size
    if j >= len(block_table_row):
        raise ValueError("position beyond the block table")
    return int(block_table_row[j]) * block_size + position % block_size


def slot_mapping(block_tables, seq_ids, positions, block_size):
    """int64 slot of each (sequence, position) pair, by ``slot_of``."""
    out = np.empty(len(seq_ids), dtype=np.int64)
    for t, (s, p) in enumerate(zip(seq_ids, positions)):
        out[t] = slot_of(block_tables[int(s)], int(p), block_size)
    return out


def kv_append(k_pool, v_pool, k, v, slots, src_dtype, cache_dtype,
              k_scale=1.0, v_scale=1.0):
    """Write each new token's K and V into its slot of the pools (in place).

    [DEV] section 1 "Why Transformers Need a KV Cache": every decode step
    computes K and V for the new token and appends them to the cache;
    section 4: the append goes into the slot the block table names.
    ``k`` and ``v`` are ``[T, n_kv_heads, head_dim]`` in ``src_dtype``;
    slot ``slots[t]`` receives row ``t`` for every KV head.  Slots outside
    ``[0, num_blocks * block_size)`` raise ValueError (nothing is written).
    """
    nb, hkv, bs, d = k_pool.shape
    slots = np.asarray(slots, dtype=np.int64)
    if np.any(slots < 0) or np.any(slots >= nb * bs):
        raise ValueError("slot out of range")
    kq = numerics.store(k, src_dtype, cache_dtype, k_scale).reshape(len(slots), hkv, d)
    vq = numerics.store(v, src_dtype, cache_dtype, v_scale).reshape(len(slots), hkv, d)
    for t, slot in enumerate(slots):
        b, off = divmod(int(slot), bs)
        k_pool[b, :, off, :] = kq[t]
        v_pool[b, :, off, :] = vq[t]


def gather_logical(pool, block_table_row, context_len, start=0):
    """Logical ``[context_len - start, n_kv_heads, head_dim]`` view of one
    sequence: its tokens at positions ``start .. context_len - 1``.

    [DEV] section 4, block-table diagram: logical block j of a sequence lives
    in physical block ``block_table_row[j]``; walking the table in order
    recovers the sequence's tokens in order.  ``start`` > 0 is a slid window
    ([VK] "A minimal PyTorch sketch", truncate): positions before it are not
    read, so their blocks may have been released.
    """
    nb, hkv, bs, d = pool.shape
    rows = []
    for t in range(int(start), int(context_len)):
        pb = int(block_table_row[t // bs])
        if not 0 <= pb < nb:
            raise ValueError("block id out of range")
        rows.append(pool[pb, :, t % bs, :])
    if not rows:
        return np.zeros((0, hkv, d), dtype=pool.dtype)
    return np.stack(rows, axis=0)
