"""Closed forms for KV-cache sizing and paged tail waste.

Test infrastructure only (see ``oracle/__init__.py``).
"""

# element sizes in bytes, by the names the cache model uses
DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1}


def kv_bytes_per_token(n_layers, n_kv_heads, head_dim, b):
    """KV-cache bytes one token occupies across all layers.

    [DEV] section 2 "The Concrete Math of KV Cache Growth": the factor 2 is
    one K and one V vector per layer and KV head, each ``head_dim`` elements
    of ``b`` bytes.  [HI] "What the KV cache is, and why it dominates memory"
    gives the same product written as 2 x Hkv x D x b x L.
    """
    for v in (n_layers, n_kv_heads, head_dim, b):
        if int(v) != v or v < 0:
            raise ValueError("sizes must be non-negative integers")
    return 2 * int(n_layers) * int(n_kv_heads) * int(head_dim) * int(b)


def blocks_for_tokens(n_tokens, block_size):
    """Physical blocks one sequence of ``n_tokens`` tokens holds.

    [DEV] section 4, "How the Architecture Works": a sequence's cache is cut
    into fixed blocks of ``block_size`` tokens and a new block is taken only
    when the previous one is full, so the count is the ceiling.
    """
    if block_size <= 0 or n_tokens < 0:
        raise ValueError("block_size > 0 and n_tokens >= 0 required")
    return -(-int(n_tokens) // int(block_size))


def tail_waste_slots(n_tokens, block_size):
    """Unused token slots in a sequence's last block.

    [DEV] section 4 "The Result" and [HI] "What 16-token blocks buy you":
    internal fragmentation is confined to the unfilled tail of the last
    block, so this is always in ``[0, block_size - 1]``.
    """
    return blocks_for_tokens(n_tokens, block_size) * int(block_size) - int(n_tokens)


def kv_bytes_for_sequences(context_lens, n_kv_heads, head_dim, b):
    """Algorithmic KV bytes one decode-attention layer reads: sum over the
    batch of ctx * 2 * Hkv * D * b (the per-token closed form with one layer).
    """
    return sum(int(c) for c in context_lens) * kv_bytes_per_token(1, n_kv_heads, head_dim, b)
