"""Pins of the prefix-cache oracle.

[DEV] section 5, 2 "Automatic Prefix Caching": a request whose tokens match a
previously computed sequence gets the existing physical blocks mapped into
its table (no new memory for the shared prefix).  Expected values come from
the published FNV-1a test vectors, from that scenario worked by hand, and
from brute force over the token lists of the inserted sequences."""

import os
import struct

import numpy as np
import pytest

from oracle import prefix_cache as pc
from oracle.allocator import AllocError, BlockAllocator

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fnv1a64.txt")


def _vectors():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        text, h = line.rsplit(None, 1)
        out.append((text.strip().strip('"').encode("ascii"), int(h, 16)))
    return out


def test_fnv1a64_published_vectors():
    vs = _vectors()
    assert len(vs) == 3
    for data, h in vs:
        assert pc.fnv1a64(data) == h


def test_block_key_is_fnv_over_parent_then_tokens():
    # the bytes packed another way: little-endian u64 parent, u32 tokens
    for parent, toks in [(0, [1, 2, 3, 4]), (0xDEADBEEF12345678, [7] * 16), (5, [2**31 - 1, 0, 65535, 9])]:
        data = struct.pack("<Q%dI" % len(toks), parent, *toks)
        assert pc.block_key(parent, toks) == pc.fnv1a64(data)


def test_keys_stand_for_whole_prefixes():
    bs = 4
    a = list(range(16))
    b = [99] + a[1:]                    # differs in block 0 only
    ka, kb, p, q = [], [], 0, 0
    for j in range(4):
        p = pc.block_key(p, a[j * bs:(j + 1) * bs])
        q = pc.block_key(q, b[j * bs:(j + 1) * bs])
        ka.append(p), kb.append(q)
    assert all(x != y for x, y in zip(ka, kb))     # block 3's tokens agree, its key does not


def _prefill(al, tokens, bs, cap=64):
    row, n = [-1] * cap, 0
    for t in range(len(tokens)):
        _, n, _ = al.append_slot(row, n, t, bs)
    return row, n


def test_system_prompt_scenario():
    # request A: 48-token system prompt (3 blocks of 16) + a 10-token question;
    # request B: the same prompt + another question.  B maps A's three prompt
    # blocks and takes no block for them.
    bs = 16
    al = BlockAllocator(32)
    cache = pc.PrefixCache(al, bs)
    prompt = list(range(1000, 1048))
    a_tokens = prompt + list(range(10))
    a_row, a_n = _prefill(al, a_tokens, bs)
    assert a_row[:4] == [0, 1, 2, 3]
    assert cache.insert(a_tokens, a_row, a_n) == 3          # the partial 4th block is not cached
    free_before = al.free_count
    b_row = [-1] * 8
    m = cache.match(prompt + [5, 6, 7], b_row)
    assert m == 3 and b_row[:3] == [0, 1, 2]
    assert al.free_count == free_before                     # no new memory for the prefix
    assert al.ref[:4] == [3, 3, 3, 1]                        # A, the cache, B; A's own block
    # a request that differs in the second block matches only the first
    c_row = [-1] * 8
    assert cache.match(prompt[:16] + [0] * 32, c_row) == 1 and c_row[0] == 0
    # a row shorter than the match stops at its capacity
    assert cache.match(prompt, [-1] * 2) == 2


def test_match_equals_brute_force_longest_shared_prefix():
    rng = np.random.default_rng(2)
    bs = 8
    al = BlockAllocator(4096)
    cache = pc.PrefixCache(al, bs)
    stems = [list(rng.integers(0, 50, 64)) for _ in range(4)]
    inserted = []
    for step in range(120):
        stem = stems[rng.integers(0, 4)]
        cut = int(rng.integers(0, 65))
        toks = [int(x) for x in stem[:cut]] + [int(x) for x in rng.integers(0, 50, int(rng.integers(0, 30)))]
        best = 0
        for other in inserted:
            k = 0
            while (k + 1) * bs <= min(len(toks), len(other)) and toks[k * bs:(k + 1) * bs] == other[k * bs:(k + 1) * bs]:
                k += 1
            best = max(best, k)
        row = [-1] * 16
        m = cache.match(toks, row)
        assert m == min(best, 16)
        # finish the request (prefill the rest) and cache it
        n = m
        for t in range(m * bs, len(toks)):
            _, n, _ = al.append_slot(row, n, t, bs)
        cache.insert(toks, row, n)
        inserted.append(toks)
        al.free_sequence(row, n)
        held = sum(al.ref)
        assert held == cache.size                       # only the cache holds blocks now
        assert al.free_count + held == 4096


def test_eviction_order_lru_then_deepest():
    bs = 4
    al = BlockAllocator(16)
    cache = pc.PrefixCache(al, bs)
    x = list(range(12))
    y = list(range(100, 108))
    xr, xn = _prefill(al, x, bs)               # blocks 0, 1, 2
    yr, yn = _prefill(al, y, bs)               # blocks 3, 4
    assert cache.insert(x, xr, xn) == 3        # tick 1
    assert cache.insert(y, yr, yn) == 2        # tick 2
    al.free_sequence(xr, xn)                   # x's blocks: only the cache holds them
    assert cache.evict(1) == 1 and al.free[-1] == 2        # oldest tick, deepest block
    assert cache.evict(5) == 2 and al.free[-2:] == [1, 0]  # y is still held by its request
    al.free_sequence(yr, yn)
    assert cache.evict(5) == 2 and al.free[-2:] == [4, 3]
    assert cache.size == 0 and al.free_count == 16


def test_verification_blocks_colliding_keys(monkeypatch):
    # every key collides: a request with other tokens must not be mapped
    monkeypatch.setattr(pc, "block_key", lambda parent, toks: 42)
    bs = 4
    al = BlockAllocator(8)
    cache = pc.PrefixCache(al, bs)
    a = [1, 2, 3, 4, 5, 6, 7, 8]
    row, n = _prefill(al, a, bs)
    assert cache.insert(a, row, n) == 1        # block 1's key (42) is taken by block 0: stop
    assert cache.match([9, 9, 9, 9], [-1] * 4) == 0
    assert cache.match(a, [-1] * 4) == 1


def test_insert_errors_change_nothing():
    al = BlockAllocator(8)
    cache = pc.PrefixCache(al, 4)
    before = al.dump()
    with pytest.raises(AllocError) as e:
        cache.insert(list(range(8)), [0, 1], 2)          # blocks 0, 1 are free
    assert e.value.status == "INVALID" and al.dump() == before and cache.size == 0
    with pytest.raises(AllocError) as e:
        cache.insert(list(range(4)), [99], 1)
    assert e.value.status == "RANGE"


def test_destroy_returns_every_block():
    al = BlockAllocator(8)
    cache = pc.PrefixCache(al, 4)
    row, n = _prefill(al, list(range(16)), 4)
    cache.insert(list(range(16)), row, n)
    al.free_sequence(row, n)
    assert al.free_count == 4
    cache.destroy()
    assert al.free_count == 8 and cache.size == 0
    assert al.free[-4:] == [0, 1, 2, 3]                   # released in insertion order
