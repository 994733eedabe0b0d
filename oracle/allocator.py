"""Physical block pool with reference counts and copy-on-write.

Test infrastructure only (see ``oracle/__init__.py``).

[DEV] section 4 "How the Architecture Works": all KV memory is one pool of
fixed-size physical blocks allocated up front; a sequence takes one block
when it starts and another each time its last block fills.  [HI]
"PagedAttention: virtual memory for attention state": a block needed by a
sequence comes from the free pool; "What 16-token blocks buy you": evicting
a sequence returns its blocks to the pool.  [DEV] section 5 "Zero-Copy
Forking": forked sequences point at the same physical blocks, each block
carrying a reference count, and the first write of a branch into a shared
block gives that branch a private copy (copy-on-write).

Readings where the pages are silent (state must match the library bit for
bit, so they are fixed here):

* the free pool is a LIFO stack.  A pool created with seed 0 hands out
  blocks 0, 1, 2, ...; with seed != 0 the hand-out order is a Fisher-Yates
  (Durstenfeld) shuffle of 0..N-1 driven by SplitMix64(seed): for
  i = N-1 down to 1, j = next() mod (i+1), swap(order[i], order[j]).
* a block whose count drops to 0 is pushed on top of the stack.
* copy-on-write is taken only when a write targets a block whose count is
  above 1: a new block is popped, the old block's count drops by one and
  the caller copies the block's contents on the device.
* errors leave the state unchanged: "OOM" (empty pool), "INVALID" (block
  not allocated, count underflow), "RANGE" (id or position out of range).
"""

MASK64 = (1 << 64) - 1


class AllocError(Exception):
    """Allocator failure; ``status`` is "OOM", "INVALID" or "RANGE"."""

    def __init__(self, status, msg=""):
        super().__init__(f"{status}: {msg}")
        self.status = status


def splitmix64_stream(seed):
    """SplitMix64 (Steele, Lea and Flood 2014): yields 64-bit outputs.

    state += 0x9E3779B97F4A7C15; z = state;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB;
    output z ^ (z >> 31)   (all arithmetic modulo 2^64).
    """
    state = seed & MASK64
    while True:
        state = (state + 0x9E3779B97F4A7C15) & MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
        yield z ^ (z >> 31)


def handout_order(num_blocks, seed):
    """Order in which a fresh pool hands out its blocks (see module doc)."""
    order = list(range(num_blocks))
    if seed:
        rng = splitmix64_stream(seed)
        for i in range(num_blocks - 1, 0, -1):
            j = next(rng) % (i + 1)
            order[i], order[j] = order[j], order[i]
    return order


class BlockAllocator:
    """Model of the library's host block allocator (same operations, same state)."""

    def __init__(self, num_blocks, seed=0):
        if num_blocks <= 0:
            raise AllocError("INVALID", "num_blocks must be positive")
        self.num_blocks = num_blocks
        # stack as a list, top at the end: the first hand-out is order[0]
        self.free = list(reversed(handout_order(num_blocks, seed)))
        self.ref = [0] * num_blocks

    # -- single blocks -------------------------------------------------
    def _check_id(self, b):
        if not 0 <= b < self.num_blocks:
            raise AllocError("RANGE", f"block {b}")

    def alloc(self):
        """Pop a free block; its count becomes 1."""
        if not self.free:
            raise AllocError("OOM", "free pool empty")
        b = self.free.pop()
        self.ref[b] = 1
        return b

    def incref(self, b):
        """One more block table points at ``b`` (fork / prefix share)."""
        self._check_id(b)
        if self.ref[b] == 0:
            raise AllocError("INVALID", f"block {b} is free")
        self.ref[b] += 1

    def decref(self, b):
        """One block table fewer points at ``b``; at 0 it returns to the pool."""
        self._check_id(b)
        if self.ref[b] == 0:
            raise AllocError("INVALID", f"block {b} is free")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            self.free.append(b)

    def cow(self, b):
        """Block to write instead of ``b``: ``(b, False)`` if private, else a
        fresh block and True (the caller copies ``b`` into it)."""
        self._check_id(b)
        if self.ref[b] == 0:
            raise AllocError("INVALID", f"block {b} is free")
        if self.ref[b] == 1:
            return b, False
        new = self.alloc()
        self.ref[b] -= 1
        return new, True

    # -- sequences -------------------------------------------------------
    def append_slot(self, table_row, num_blocks, position, block_size):
        """Slot for writing logical token ``position`` of a sequence.

        ``table_row`` is the sequence's block table (a mutable list whose
        length is the table capacity) holding ``num_blocks`` valid entries.
        A position just past the last block takes a new block; a position
        inside a shared block takes a private copy first.  Returns
        ``(slot, num_blocks, cow)`` where ``cow`` is ``(src, dst)`` or None.
        """
        cap = len(table_row)
        if position < 0 or position > num_blocks * block_size:
            raise AllocError("RANGE", f"position {position}")
        j = position // block_size
        cow = None
        if j == num_blocks:
            if j >= cap:
                raise AllocError("RANGE", "block table full")
            table_row[j] = self.alloc()
            num_blocks += 1
        else:
            b = table_row[j]
            new, copied = self.cow(b)
            if copied:
                table_row[j] = new
                cow = (b, new)
        return table_row[j] * block_size + position % block_size, num_blocks, cow

    def fork(self, table_row, num_blocks):
        """Share every block of a sequence with a new branch (count + 1 each).

        All or nothing: a bad id undoes the increments already made."""
        done = []
        try:
            for b in table_row[:num_blocks]:
                self.incref(b)
                done.append(b)
        except AllocError:
            for b in done:
                self.ref[b] -= 1
            raise

    def free_sequence(self, table_row, num_blocks):
        """Drop a sequence: decref its blocks in table order.

        All or nothing: every id is checked (in range, referenced as often as
        the row names it) before any count changes."""
        uses = {}
        for b in table_row[:num_blocks]:
            self._check_id(b)
            uses[b] = uses.get(b, 0) + 1
            if self.ref[b] < uses[b]:
                raise AllocError("INVALID", f"block {b} over-released")
        for b in table_row[:num_blocks]:
            self.decref(b)

    def truncate(self, table_row, num_blocks, start, length, keep, block_size):
        """Slide a sequence's window so that only its last ``keep`` tokens stay.

        [VK] "PagedAttention: the idea": when the window slides, the oldest
        page goes back to the allocator.  [VK] "A minimal PyTorch sketch",
        ``truncate`` and the notes under it: whole pages are dropped first and
        what remains of the drop is an offset into the first kept page, with
        no copy.  The sketch records that offset only by shortening the
        length, which would make later reads return the wrong rows; the
        reading taken here keeps an explicit start instead.

        The sequence occupies row positions ``[start, length)`` (position p
        in ``table_row[p // block_size]``, offset ``p % block_size``).  The
        new start is ``max(start, length - keep)``; every block whose
        positions all lie before it is released (``decref``, row order) and
        removed from the front of the row, the remaining ids move to the
        front and the freed tail entries become -1.  Positions then count
        from the first remaining block.  Returns ``(num_blocks, start,
        length)``.  All or nothing: bad arguments or ids change no state.
        """
        if keep < 0 or start < 0 or start > length or length > num_blocks * block_size \
                or num_blocks > len(table_row):
            raise AllocError("RANGE", "bad window")
        new_start = max(start, length - keep)
        drop = new_start // block_size
        uses = {}
        for b in table_row[:drop]:
            self._check_id(b)
            uses[b] = uses.get(b, 0) + 1
            if self.ref[b] < uses[b]:
                raise AllocError("INVALID", f"block {b} over-released")
        for b in table_row[:drop]:
            self.decref(b)
        kept = list(table_row[drop:num_blocks])
        table_row[:num_blocks] = kept + [-1] * drop
        return num_blocks - drop, new_start - drop * block_size, length - drop * block_size

    # -- state -----------------------------------------------------------
    @property
    def free_count(self):
        return len(self.free)

    def dump(self):
        """``(free stack bottom-to-top, refcounts)`` for bit-exact comparison."""
        return list(self.free), list(self.ref)
