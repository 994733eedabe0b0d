"""Single-query (decode) attention over a contiguous or a paged KV cache.

Test infrastructure only (see ``oracle/__init__.py``).

[DEV] section 1 "Why Transformers Need a KV Cache" defines attention as
softmax(Q K^T / sqrt(d_k)) V; at decode time the query is the one new token
and K, V are every cached token of the sequence.  [DEV] section 2, Example 2
(grouped-query attention): several query heads share one KV head.  Reading
taken for the grouping: query head ``h`` uses KV head ``h // G`` with
``G = n_q_heads / n_kv_heads`` (consecutive groups).  The softmax scale is a
parameter (the pages' 1/sqrt(d_k) is what the workloads pass).

Everything is computed in float64 from exactly-widened inputs, with the
maximum score subtracted before exponentiation.  A sequence with no cached
token has output 0 (the pages say nothing; this is our reading).
"""

import numpy as np

from . import cache, numerics


def decode_attention_contiguous(q, K, V, scale):
    """Output ``[n_q_heads, head_dim]`` for one sequence.

    ``q`` is ``[n_q_heads, head_dim]``; ``K`` and ``V`` are
    ``[context_len, n_kv_heads, head_dim]`` in logical token order; all are
    float64 (or exactly widened to it).
    """
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, d = q.shape
    ctx, hkv, _ = K.shape
    if hq % hkv:
        raise ValueError("n_q_heads must be a multiple of n_kv_heads")
    g = hq // hkv
    out = np.zeros((hq, d), dtype=np.float64)
    if ctx == 0:
        return out
    for h in range(hq):
        kv = h // g
        s = (K[:, kv, :] @ q[h]) * float(scale)     # one score per cached token
        w = np.exp(s - s.max())
        out[h] = (w @ V[:, kv, :]) / w.sum()
    return out


def decode_attention_paged(q, k_pool, v_pool, block_tables, context_lens, scale,
                           kv_dtype, k_scale=1.0, v_scale=1.0, q_dtype="f32", context_starts=None):
    """Output ``[batch, n_q_heads, head_dim]`` (float64) of paged decode attention.

    [DEV] section 4 "The PagedAttention CUDA Kernel": for each sequence the
    kernel reads the query, looks the sequence's blocks up in its block table
    and fetches K and V from the scattered physical blocks.  Here that is the
    logical gather of ``oracle.cache.gather_logical`` followed by the
    contiguous definition above, on the exactly dequantised cache values
    (``decode(code) * scale`` for FP8).  ``context_starts`` (one per
    sequence, default 0) restricts sequence s to the positions
    ``context_starts[s] .. context_lens[s] - 1`` of its row: a window slid by
    truncation ([VK] "A minimal PyTorch sketch"); an empty window gives 0.
    """
    qf = numerics.to_f64(q, q_dtype)
    batch = qf.shape[0]
    out = np.zeros(qf.shape, dtype=np.float64)
    for s in range(batch):
        ctx = int(context_lens[s])
        st = 0 if context_starts is None else min(int(context_starts[s]), ctx)
        Kr = cache.gather_logical(k_pool, block_tables[s], ctx, st)
        Vr = cache.gather_logical(v_pool, block_tables[s], ctx, st)
        K = numerics.to_f64(Kr, kv_dtype, k_scale)
        V = numerics.to_f64(Vr, kv_dtype, v_scale)
        out[s] = decode_attention_contiguous(qf[s], K, V, scale)
    return out
