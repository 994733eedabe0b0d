"""Pins for oracle.allocator: the copy-on-write scenario printed on the pages, the
75% prompt-memory claim, the published SplitMix64 outputs, hand-written traces
and the conservation invariant."""

import os

import numpy as np
import pytest

from oracle.allocator import AllocError, BlockAllocator, handout_order, splitmix64_stream

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cow_fixture():
    with open(os.path.join(GOLDEN, "cow_scenario.txt")) as f:
        kv = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    return {r[0]: [int(x) for x in r[1:]] for r in kv}


def test_splitmix64_published_outputs():
    # first outputs of SplitMix64 seeded with 1234567 (the generator's published
    # reference implementation)
    g = splitmix64_stream(1234567)
    assert [next(g) for _ in range(5)] == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_fresh_pool_hands_out_in_order():
    a = BlockAllocator(5)
    assert [a.alloc() for _ in range(5)] == [0, 1, 2, 3, 4]
    with pytest.raises(AllocError) as e:
        a.alloc()
    assert e.value.status == "OOM"
    assert a.free_count == 0


def test_seeded_order_is_a_permutation_and_is_used():
    order = handout_order(1000, 42)
    assert sorted(order) == list(range(1000)) and order != list(range(1000))
    a = BlockAllocator(1000, seed=42)
    assert [a.alloc() for _ in range(10)] == order[:10]
    # small case by hand: N=3, draws r1 (i=2) and r2 (i=1) from SplitMix64(42)
    g = splitmix64_stream(42)
    r1, r2 = next(g), next(g)
    o = [0, 1, 2]
    j = r1 % 3
    o[2], o[j] = o[j], o[2]
    j = r2 % 2
    o[1], o[j] = o[j], o[1]
    assert handout_order(3, 42) == o


def test_hand_trace_lifo_stack():
    a = BlockAllocator(4)
    b0, b1, b2 = a.alloc(), a.alloc(), a.alloc()
    assert (b0, b1, b2) == (0, 1, 2)
    a.decref(1)
    assert a.dump() == ([3, 1], [1, 0, 1, 0])
    a.incref(0)
    a.decref(0)
    assert a.dump() == ([3, 1], [1, 0, 1, 0])
    a.decref(0)
    assert a.dump() == ([3, 1, 0], [0, 0, 1, 0])
    assert a.alloc() == 0 and a.alloc() == 1 and a.alloc() == 3
    with pytest.raises(AllocError) as e:
        a.decref(0) or a.decref(0)
    assert e.value.status == "INVALID"
    with pytest.raises(AllocError) as e:
        a.incref(4)
    assert e.value.status == "RANGE"


def test_cow_scenario_from_the_page():
    fx = _cow_fixture()
    p0, p1 = fx["prompt_blocks"]
    a_id, b_id = fx["branch_a_private"][0], fx["branch_b_private"][0]
    n = 128
    a = BlockAllocator(n)
    every = [a.alloc() for _ in range(n)]
    # return every block, the four named ones last so they are handed out first
    named = [p0, p1, a_id, b_id]
    for blk in every:
        if blk not in named:
            a.decref(blk)
    for blk in reversed(named):
        a.decref(blk)
    bs = 16
    prompt = [-1] * 4
    nblk = 0
    for pos in range(32):                       # tokens 0-31 of the prompt
        _, nblk, cow = a.append_slot(prompt, nblk, pos, bs)
        assert cow is None
    assert prompt[:2] == [p0, p1]
    a.fork(prompt, nblk)                        # a second branch shares the prompt
    assert a.ref[p0] == a.ref[p1] == fx["prompt_refcount"][0]
    branch_a, branch_b = list(prompt), list(prompt)
    slot_a, na, cow_a = a.append_slot(branch_a, nblk, 32, bs)
    slot_b, nb_, cow_b = a.append_slot(branch_b, nblk, 32, bs)
    assert branch_a[2] == a_id and branch_b[2] == b_id
    assert (slot_a, slot_b) == (a_id * bs, b_id * bs)
    assert cow_a is None and cow_b is None      # full shared blocks are never written
    assert branch_a[:2] == branch_b[:2] == [p0, p1]


def test_cow_on_a_partly_filled_shared_block():
    a = BlockAllocator(10)
    row = [-1] * 4
    n = 0
    for pos in range(20):                       # block 0 full, block 1 holds 4 tokens
        _, n, _ = a.append_slot(row, n, pos, 16)
    a.fork(row, n)
    child = list(row)
    slot, n2, cow = a.append_slot(child, n, 20, 16)
    assert cow == (1, 2) and child[1] == 2 and slot == 2 * 16 + 4
    assert a.ref[1] == 1 and a.ref[2] == 1 and a.ref[0] == 2
    # the parent writes its own next token in place: its block is now private
    slot_p, _, cow_p = a.append_slot(row, n, 20, 16)
    assert cow_p is None and slot_p == 1 * 16 + 4


def test_four_branches_cut_prompt_memory_by_75_percent():
    fx = _cow_fixture()
    branches = fx["branches_for_75_percent"][0]
    a = BlockAllocator(256)
    prompt = [-1] * 16
    n = 0
    for pos in range(16 * 10):                  # a 10-block prompt
        _, n, _ = a.append_slot(prompt, n, pos, 16)
    for _ in range(branches - 1):
        a.fork(prompt, n)
    used = 256 - a.free_count
    naive = branches * n
    assert used == n and 1 - used / naive == 0.75


def test_errors_leave_state_unchanged():
    a = BlockAllocator(2)
    row = [-1]
    _, n, _ = a.append_slot(row, 0, 0, 16)
    state = a.dump()
    for call in (lambda: a.append_slot(row, n, 16, 16),   # table full
                 lambda: a.append_slot(row, n, 40, 16),   # gap in positions
                 lambda: a.decref(1)):
        with pytest.raises(AllocError):
            call()
        assert a.dump() == state
    a.fork(row, n)
    a.alloc()                                             # pool now empty
    state = a.dump()
    with pytest.raises(AllocError) as e:
        a.append_slot(list(row), n, 3, 16)               # CoW needs a block
    assert e.value.status == "OOM" and a.dump() == state


def test_random_trace_conserves_blocks():
    rng = np.random.default_rng(0)
    a = BlockAllocator(64, seed=7)
    held = []
    for _ in range(5000):
        op = rng.integers(0, 3)
        try:
            if op == 0:
                held.append(a.alloc())
            elif op == 1 and held:
                b = held[rng.integers(len(held))]
                a.incref(b)
                held.append(b)
            elif held:
                b = held.pop(rng.integers(len(held)))
                a.decref(b)
        except AllocError as e:
            assert e.status == "OOM"
        free, ref = a.dump()
        assert len(set(free)) == len(free)
        assert all(ref[b] == 0 for b in free)
        assert sum(1 for r in ref if r > 0) + len(free) == 64
        assert sum(ref) == len(held)
