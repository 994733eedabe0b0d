"""Pins of the sliding-window oracle: allocator truncate and windowed attention.

[VK] "PagedAttention: the idea": sliding the window returns the oldest page
to the allocator.  [VK] "A minimal PyTorch sketch", truncate: whole pages go
first, the rest of the drop is an offset into the first kept page, no copy.
The expected values below come from that rule worked by hand, from a plain
list model of each sequence's token stream, and from the contiguous
attention definition on slices of the unpaged arrays.
"""

import numpy as np
import pytest

from oracle import allocator, attention, cache
from oracle.allocator import AllocError


def _ids_pool(num_blocks, bs):
    """A pool whose every slot will hold the id of the token written there."""
    return np.full((num_blocks, 1, bs, 1), -1, dtype=np.int64)


def _write(pool, al, row, nblk, pos, token_id, bs):
    slot, nblk, cow = al.append_slot(row, nblk, pos, bs)
    if cow is not None:
        pool[cow[1]] = pool[cow[0]]
    b, off = divmod(slot, bs)
    pool[b, 0, off, 0] = token_id
    return nblk


def test_page_example_600_tokens_keep_300():
    # 256-token pages as in the sketch: 600 tokens fill pages of 256, 256, 88.
    # Keeping the last 300 drops 300 tokens: one whole page (256) is released
    # and the remaining 44 become the offset into the first kept page.
    bs = 256
    al = allocator.BlockAllocator(8)
    row, nblk = [-1] * 4, 0
    pool = _ids_pool(8, bs)
    for t in range(600):
        nblk = _write(pool, al, row, nblk, t, t, bs)
    assert row == [0, 1, 2, -1] and nblk == 3
    nblk, start, length = al.truncate(row, nblk, 0, 600, 300, bs)
    assert (nblk, start, length) == (2, 44, 344)
    assert row == [1, 2, -1, -1]
    assert al.ref[0] == 0 and al.free_count == 6
    got = cache.gather_logical(pool, row, length, start)[:, 0, 0]
    assert list(got) == list(range(300, 600))


def test_released_blocks_go_back_in_row_order():
    # LIFO pool: blocks 0 and 1 are pushed in row order, so 1 comes out first
    bs = 16
    al = allocator.BlockAllocator(4)
    row, nblk = [-1] * 4, 0
    pool = _ids_pool(4, bs)
    for t in range(40):
        nblk = _write(pool, al, row, nblk, t, t, bs)
    nblk, start, length = al.truncate(row, nblk, 0, 40, 5, bs)   # new start 35: blocks 0, 1 go
    assert (nblk, start, length, row) == (1, 3, 8, [2, -1, -1, -1])
    assert al.alloc() == 1 and al.alloc() == 0


def test_shared_blocks_lose_one_reference_only():
    bs = 16
    al = allocator.BlockAllocator(8)
    a, na = [-1] * 4, 0
    pool = _ids_pool(8, bs)
    for t in range(40):
        na = _write(pool, al, a, na, t, t, bs)
    b = list(a)
    al.fork(b, na)                                   # b shares blocks 0, 1, 2
    na, sa, la = al.truncate(a, na, 0, 40, 10, bs)   # a's start 30: drops 0
    assert (na, sa, la) == (2, 14, 24)
    assert al.ref[:3] == [1, 2, 2] and al.free_count == 5
    assert list(cache.gather_logical(pool, b, 40)[:, 0, 0]) == list(range(40))   # b unaffected
    assert list(cache.gather_logical(pool, a, la, sa)[:, 0, 0]) == list(range(30, 40))


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_random_traces_match_a_token_list_model(bs):
    """Appends, truncations, forks and frees on several sequences; after every
    step each window holds exactly its list model's tokens, and references
    add up (free blocks + referenced blocks = pool; sum of counts = row entries)."""
    rng = np.random.default_rng(7 + bs)
    nb = 64
    al = allocator.BlockAllocator(nb, seed=5)
    pool = _ids_pool(nb, bs)
    seqs = []   # [row, nblk, start, length, model tokens]
    next_id = 0
    for step in range(400):
        op = rng.integers(0, 10)
        if op < 6 or not seqs:                       # append to a sequence (new or existing)
            if not seqs or rng.integers(0, 8) == 0:
                seqs.append([[-1] * 40, 0, 0, 0, []])
            sq = seqs[rng.integers(0, len(seqs))]
            try:
                sq[1] = _write(pool, al, sq[0], sq[1], sq[3], next_id, bs)
            except AllocError:
                continue
            sq[3] += 1
            sq[4].append(next_id)
            next_id += 1
        elif op < 8:                                 # slide a window
            sq = seqs[rng.integers(0, len(seqs))]
            keep = int(rng.integers(0, 3 * bs))
            sq[1], sq[2], sq[3] = al.truncate(sq[0], sq[1], sq[2], sq[3], keep, bs)
            if keep < len(sq[4]):
                sq[4] = sq[4][len(sq[4]) - keep:]
        elif op < 9:                                 # fork
            src = seqs[rng.integers(0, len(seqs))]
            try:
                al.fork(src[0], src[1])
            except AllocError:
                continue
            seqs.append([list(src[0]), src[1], src[2], src[3], list(src[4])])
        else:                                        # free a sequence
            sq = seqs.pop(rng.integers(0, len(seqs)))
            al.free_sequence(sq[0], sq[1])
        refs = sum(1 for s in seqs for b in s[0][:s[1]])
        assert sum(al.ref) == refs
        assert al.free_count + sum(1 for r in al.ref if r > 0) == nb
        for row, nblk, start, length, model in seqs:
            assert 0 <= start <= length <= nblk * bs and start < bs
            got = cache.gather_logical(pool, row, length, start)[:, 0, 0]
            assert list(got) == model


def test_truncate_errors_change_nothing():
    bs = 16
    al = allocator.BlockAllocator(4)
    row, nblk = [-1] * 4, 0
    for t in range(20):
        _, nblk, _ = al.append_slot(row, nblk, t, bs)
    before = al.dump(), list(row)
    for args in [(row, nblk, 0, 20, -1), (row, nblk, 21, 20, 5), (row, nblk, 0, 40, 5)]:
        with pytest.raises(AllocError) as e:
            al.truncate(*args, bs)
        assert e.value.status == "RANGE"
    bad = [3, 0, -1, -1]                 # block 3 is free: releasing it would underflow
    with pytest.raises(AllocError) as e:
        al.truncate(bad, 2, 0, 32, 4, bs)
    assert e.value.status == "INVALID"
    assert (al.dump(), list(row)) == before
    assert al.truncate(row, nblk, 0, 20, 20, bs) == (2, 0, 20)    # keep everything
    assert al.truncate(row, nblk, 0, 20, 0, bs) == (1, 4, 4)      # empty window: start == length


def _random_kv(rng, n, hkv, d):
    """float32 draws, held in float64 (exact)"""
    return (rng.standard_normal((n, hkv, d)).astype(np.float32).astype(np.float64),
            rng.standard_normal((n, hkv, d)).astype(np.float32).astype(np.float64))


def test_windowed_attention_is_attention_over_the_tail():
    rng = np.random.default_rng(3)
    bs, hkv, hq, d = 16, 2, 4, 8
    ctxs, starts = [50, 33, 16, 7], [13, 0, 16, 3]
    nb = 16
    perm = rng.permutation(nb)
    kp = np.full((nb, hkv, bs, d), np.nan, dtype=np.float32)
    vp = np.full((nb, hkv, bs, d), np.nan, dtype=np.float32)
    tables = np.full((4, 4), -1, dtype=np.int64)
    q = rng.standard_normal((4, hq, d)).astype(np.float32).astype(np.float64)
    want = np.zeros((4, hq, d))
    used = 0
    for s, (ctx, st) in enumerate(zip(ctxs, starts)):
        K, V = _random_kv(rng, ctx, hkv, d)
        for j in range(-(-ctx // bs)):
            if (j + 1) * bs <= st:
                continue                              # released block: stays -1 and NaN
            tables[s, j] = perm[used]
            used += 1
            for t in range(j * bs, min(ctx, (j + 1) * bs)):
                kp[tables[s, j], :, t % bs] = K[t]
                vp[tables[s, j], :, t % bs] = V[t]
        # the definition on the tail of the unpaged arrays, written out
        for h in range(hq):
            kv = h // (hq // hkv)
            sc = K[st:, kv] @ q[s, h] * 0.3
            if len(sc):
                w = np.exp(sc - sc.max())
                want[s, h] = w @ V[st:, kv] / w.sum()
    got = attention.decode_attention_paged(q, kp, vp, tables, ctxs, 0.3, "f32", context_starts=starts)
    assert np.allclose(got, want, rtol=0, atol=1e-12)
    assert np.all(got[2] == 0)                        # start == ctx: empty window


def test_window_after_truncate_equals_attention_over_the_last_tokens():
    rng = np.random.default_rng(11)
    bs, hkv, hq, d, n, keep = 16, 1, 2, 8, 100, 37
    K, V = _random_kv(rng, n, hkv, d)
    q = rng.standard_normal((1, hq, d)).astype(np.float32).astype(np.float64)
    al = allocator.BlockAllocator(10, seed=9)
    row, nblk = [-1] * 8, 0
    kp = np.full((10, hkv, bs, d), np.nan, dtype=np.float32)
    vp = np.full((10, hkv, bs, d), np.nan, dtype=np.float32)
    for t in range(n):
        slot, nblk, _ = al.append_slot(row, nblk, t, bs)
        kp[slot // bs, :, slot % bs] = K[t]
        vp[slot // bs, :, slot % bs] = V[t]
    nblk, start, length = al.truncate(row, nblk, 0, n, keep, bs)
    assert length - start == keep
    got = attention.decode_attention_paged(q, kp, vp, np.array([row]), [length], 0.25, "f32",
                                           context_starts=[start])
    want = attention.decode_attention_contiguous(q[0], K[n - keep:], V[n - keep:], 0.25)
    assert np.array_equal(got[0], want)
