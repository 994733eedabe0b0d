"""Automatic prefix caching: a hash table of full KV blocks keyed by prefix.

Test infrastructure only (see ``oracle/__init__.py``).

[DEV] section 5 "Superpowers of Paged Memory", 2 "Automatic Prefix Caching":
when a new request's tokens match a previously computed sequence, the engine
looks its blocks up in a hash table of physical blocks and, where the tokens
match, maps the existing blocks into the new request's block table instead
of computing them again; the shared prefix then costs no extra memory.
[HI] "Prefix caching: share the system prompt": one copy of the prefix KV,
mapped into every request's table.

The pages fix neither the hash nor the table's policies.  Readings taken:

* only full blocks are cached (a block still being filled may change);
* block j of a token sequence has the key
  ``K_j = FNV-1a-64(LE64(K_{j-1}) || LE32(t_{j*bs}) || ... || LE32(t_{j*bs+bs-1}))``
  with ``K_{-1} = 0``, so a key stands for the whole prefix up to its block;
  FNV-1a-64 is the published Fowler-Noll-Vo function (offset basis
  0xcbf29ce484222325, prime 0x100000001b3: for each byte, xor then multiply
  modulo 2^64);
* a lookup hit is verified: the entry's parent key and token ids must equal
  the request's, so a hash collision never maps a wrong block; an insert
  that meets an entry with other contents under its key stops there;
* the cache holds one reference on each cached block (so it outlives the
  request that computed it); a match takes one more reference per mapped
  block for the new request;
* eviction releases entries that only the cache still references, least
  recently used first (all blocks of one match or insert share one tick),
  deeper blocks first within a tick, then by key;
* destroying the cache releases its references in insertion order.
"""

from .allocator import AllocError

MASK64 = (1 << 64) - 1
FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3


def fnv1a64(data, h=FNV_OFFSET):
    """FNV-1a, 64 bits, over a bytes-like object."""
    for b in bytes(data):
        h = ((h ^ b) * FNV_PRIME) & MASK64
    return h


def block_key(parent_key, block_tokens):
    """Key of a full block given its parent's key and its token ids."""
    data = int(parent_key & MASK64).to_bytes(8, "little")
    for t in block_tokens:
        data += int(t & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


class PrefixCache:
    """Model of the library's prefix cache over an ``oracle.allocator.BlockAllocator``."""

    def __init__(self, allocator, block_size):
        if block_size <= 0:
            raise ValueError("block_size must be positive")
        self.al = allocator
        self.bs = block_size
        # key -> dict(block, parent, tokens, depth, tick, order)
        self.entries = {}
        self.cached_blocks = set()
        self.tick = 0
        self.order = 0

    @property
    def size(self):
        return len(self.entries)

    def _walk(self, tokens, n_blocks):
        """(key, parent key, token tuple) of the first n_blocks full blocks."""
        parent = 0
        for j in range(n_blocks):
            blk = tuple(int(t) for t in tokens[j * self.bs:(j + 1) * self.bs])
            key = block_key(parent, blk)
            yield j, key, parent, blk
            parent = key

    def match(self, tokens, table_row):
        """Map the longest cached full-block prefix of ``tokens`` into
        ``table_row`` (a list, at most its length); returns the blocks matched."""
        self.tick += 1
        n = min(len(tokens) // self.bs, len(table_row))
        m = 0
        for j, key, parent, blk in self._walk(tokens, n):
            e = self.entries.get(key)
            if e is None or e["parent"] != parent or e["tokens"] != blk:
                break
            self.al.incref(e["block"])
            table_row[j] = e["block"]
            e["tick"] = self.tick
            m += 1
        return m

    def insert(self, tokens, table_row, num_blocks):
        """Cache the full blocks of a computed sequence (its row holds
        ``num_blocks`` valid ids); returns how many new entries were made.

        All or nothing: an id that is out of range or free raises before any
        change."""
        n = min(num_blocks, len(tokens) // self.bs)
        plan, planned = [], {}
        for j, key, parent, blk in self._walk(tokens, n):
            e = self.entries.get(key, planned.get(key))
            if e is not None:
                if e["parent"] != parent or e["tokens"] != blk:
                    break                      # collision: keep the owner's chain
                plan.append(("touch", key, None))
                continue
            b = int(table_row[j])
            if b in self.cached_blocks or any(p[0] == "new" and p[2]["block"] == b for p in plan):
                break                          # a block is cached under one key at most
            self.al._check_id(b)
            if self.al.ref[b] == 0:
                raise AllocError("INVALID", f"block {b} is free")
            planned[key] = {"block": b, "parent": parent, "tokens": blk, "depth": j}
            plan.append(("new", key, planned[key]))
        self.tick += 1
        made = 0
        for kind, key, e in plan:
            if kind == "touch":
                self.entries[key]["tick"] = self.tick
                continue
            self.al.incref(e["block"])
            e["tick"] = self.tick
            e["order"] = self.order
            self.order += 1
            self.entries[key] = e
            self.cached_blocks.add(e["block"])
            made += 1
        return made

    def evict(self, max_blocks):
        """Release up to ``max_blocks`` entries only the cache references;
        returns how many were released."""
        cands = [(e["tick"], -e["depth"], key) for key, e in self.entries.items()
                 if self.al.ref[e["block"]] == 1]
        cands.sort()
        done = 0
        for _, _, key in cands[:max(0, max_blocks)]:
            e = self.entries.pop(key)
            self.cached_blocks.discard(e["block"])
            self.al.decref(e["block"])
            done += 1
        return done

    def destroy(self):
        for key, e in sorted(self.entries.items(), key=lambda kv: kv[1]["order"]):
            self.al.decref(e["block"])
        self.entries.clear()
        self.cached_blocks.clear()
