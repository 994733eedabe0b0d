"""Split-context decode attention: per-partition partials and their merge.

Test infrastructure only (see ``oracle/__init__.py``).

The pages stop at the single-pass kernel; splitting a long context into
fixed partitions whose partial softmax states are merged afterwards is the
flash-decoding arrangement the long-context workload ([HI] "Why this matters
for long context") needs to keep a GPU busy.  Partition ``p`` of a sequence
covers logical tokens ``[p*P, min((p+1)*P, ctx))``.  Each partition yields,
per query head, its score maximum ``m``, the sum ``l`` of ``exp(s - m)``
and its normalised output ``o``; the merge

    M = max_p m_p,   w_p = l_p * exp(m_p - M),   out = sum_p w_p o_p / sum_p w_p

is exactly the softmax over the whole context, so the result equals
``attention.decode_attention_contiguous`` up to float64 rounding.
"""

import numpy as np


def partition_partials(q, K, V, scale, partition_size):
    """``(m, l, o)`` of each partition: shapes ``[P, Hq]``, ``[P, Hq]``, ``[P, Hq, D]``."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    hq, d = q.shape
    ctx, hkv, _ = K.shape
    g = hq // hkv
    n_part = max(1, -(-ctx // partition_size))
    m = np.full((n_part, hq), -np.inf)
    l = np.zeros((n_part, hq))
    o = np.zeros((n_part, hq, d))
    for p in range(n_part):
        lo, hi = p * partition_size, min((p + 1) * partition_size, ctx)
        if hi <= lo:
            continue
        for h in range(hq):
            kv = h // g
            s = (K[lo:hi, kv, :] @ q[h]) * float(scale)
            m[p, h] = s.max()
            w = np.exp(s - m[p, h])
            l[p, h] = w.sum()
            o[p, h] = (w @ V[lo:hi, kv, :]) / l[p, h]
    return m, l, o


def merge_partials(m, l, o):
    """Merge partition partials into the final ``[Hq, D]`` output (see module doc)."""
    m = np.asarray(m, dtype=np.float64)
    l = np.asarray(l, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    n_part, hq, d = o.shape
    out = np.zeros((hq, d))
    for h in range(hq):
        M = m[:, h].max()
        if not np.isfinite(M):
            continue                        # no token at all: output 0
        w = l[:, h] * np.exp(m[:, h] - M)
        out[h] = (w[:, None] * o[:, h, :]).sum(axis=0) / w.sum()
    return out


def decode_attention_split(q, K, V, scale, partition_size):
    """Split-context decode attention of one sequence (float64)."""
    return merge_partials(*partition_partials(q, K, V, scale, partition_size))
