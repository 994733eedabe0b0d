"""The synthetic decode workloads: shapes, context lengths, block tables, values.

Each workload is seeded by its index (``seed``) and drawn from streams of
``synth`` that are independent per tensor and per sequence, so one
sequence's K/V can be drawn without drawing the rest.  Only numbers and
layouts come from here; slots, appends, quantisation, allocation and
attention are computed by each side on its own.

Workloads (values ~N(0,1) throughout, block size 16 unless noted):

* ``tiny``      4 sequences, contexts {5, 17, 33, 64}; Hq=4, Hkv=2, D=64,
                float32 Q/K/V; pool of 32 blocks, the 10 blocks used are the
                first 10 of a seeded permutation of 0..31; scale 1/8.
* ``gqa_bf16``  Llama-3-8B-shaped layer: Hq=32, Hkv=8, D=128, bfloat16;
                batch 32, contexts uniform in [1, 4096]; the pool holds
                exactly the blocks in use plus 32 spare, block tables are a
                shuffled partition of it; a 32-token append goes to 32
                distinct slots drawn from the pool's unused slots.
* ``mha_f16``   Llama-2-13B-shaped layer: Hq=Hkv=40, D=128, float16; batch
                8, every context 4096; 2048 blocks, shuffled.
* ``prefix_bf16`` prefix sharing: Hq=32, Hkv=8, D=128, bfloat16; batch 64; a
                2048-token prefix (128 blocks) shared by every sequence, plus
                private suffixes of length uniform in [1, 512]; allocation
                goes through the block allocator (a seeded hand-out order),
                and each sequence appends one token before decoding.
* ``longctx_fp8`` 70B-shaped long context: Hq=64, Hkv=8, D=128; K/V stored as
                FP8 E4M3 with one float32 scale per cache tensor (the largest
                |value| of that tensor / 448), bfloat16 Q; batch 4, every
                context 131072; 32768 blocks, shuffled; partitions of 512.
"""

import dataclasses
import math

import numpy as np

from . import normal_f32, permutation, sample_without_replacement, uniform_int

# stream ids (upper bits: tensor; lower 32 bits: sequence)
S_Q, S_K, S_V, S_CTX, S_PERM, S_APPEND_SLOTS, S_APPEND_K, S_APPEND_V = range(1, 9)
S_PREFIX_K, S_PREFIX_V, S_SUFFIX = 9, 10, 11


def _stream(tensor, seq=0):
    return (tensor << 32) | seq


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    batch: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    block_size: int
    kv_dtype: str            # "f32" | "f16" | "bf16" | "fp8_e4m3"
    q_dtype: str             # "f32" | "f16" | "bf16"
    scale: float
    partition_size: int      # tokens per split-context partition, 0 = library's choice
    context_lens: np.ndarray  # int32 [batch]: tokens already cached before the step
    num_blocks: int
    block_tables: np.ndarray | None   # int32 [batch, max_blocks] (None: via allocator)
    max_blocks: int
    append_tokens: int = 0           # new tokens appended in one step
    prefix_len: int = 0              # shared prefix tokens (prefix workload)
    alloc_seed: int = 0              # allocator hand-out seed (prefix workload)

    @property
    def group(self):
        return self.n_q_heads // self.n_kv_heads

    @property
    def kv_elem_bytes(self):
        return {"f32": 4, "f16": 2, "bf16": 2, "fp8_e4m3": 1}[self.kv_dtype]

    @property
    def src_dtype(self):
        """Type of the new-token K/V handed to append (float32 before FP8)."""
        return "f32" if self.kv_dtype == "fp8_e4m3" else self.kv_dtype


NAMES = ("tiny", "gqa_bf16", "mha_f16", "prefix_bf16", "longctx_fp8")


def _shuffled_tables(seed, ctx, bs, num_blocks, max_blocks):
    """Deal a seeded permutation of the pool out to the sequences in order."""
    perm = permutation(seed, _stream(S_PERM), num_blocks)
    tables = np.zeros((len(ctx), max_blocks), dtype=np.int32)
    pos = 0
    for s, c in enumerate(ctx):
        n = -(-int(c) // bs)
        tables[s, :n] = perm[pos:pos + n]
        pos += n
    return tables


def make(name, block_size=None):
    """The workload called ``name`` (small metadata only; values are drawn lazily).

    ``block_size`` (8, 16 or 32) re-blocks the gqa_bf16, mha_f16 and
    longctx_fp8 workloads; token values, context lengths and pool bytes stay
    the same (the default is their 16-token blocks)."""
    seed = NAMES.index(name)
    if block_size not in (None, 16) and name not in ("gqa_bf16", "mha_f16", "longctx_fp8"):
        raise ValueError(f"{name} has 16-token blocks only")
    bs_x = block_size or 16
    if name == "tiny":
        ctx = np.array([5, 17, 33, 64], dtype=np.int32)
        return Workload(name, seed, 4, 4, 2, 64, 16, "f32", "f32", 1.0 / 8.0, 0, ctx, 32,
                        _shuffled_tables(seed, ctx, 16, 32, 4), 4)
    if name == "gqa_bf16":
        b, bs = 32, bs_x
        ctx = uniform_int(seed, _stream(S_CTX), b, 1, 4096).astype(np.int32)
        used = sum(-(-int(c) // bs) for c in ctx)
        nb = used + 32 * 16 // bs
        return Workload(name, seed, b, 32, 8, 128, bs, "bf16", "bf16", 1 / math.sqrt(128), 0,
                        ctx, nb, _shuffled_tables(seed, ctx, bs, nb, 4096 // bs), 4096 // bs,
                        append_tokens=32)
    if name == "mha_f16":
        b, bs = 8, bs_x
        ctx = np.full(b, 4096, dtype=np.int32)
        nb = b * 4096 // bs
        return Workload(name, seed, b, 40, 40, 128, bs, "f16", "f16", 1 / math.sqrt(128), 0,
                        ctx, nb, _shuffled_tables(seed, ctx, bs, nb, 4096 // bs), 4096 // bs)
    if name == "prefix_bf16":
        b, bs, prefix = 64, 16, 2048
        suffix = uniform_int(seed, _stream(S_SUFFIX), b, 1, 512)
        ctx = (prefix + suffix).astype(np.int32)
        private = sum(-(-int(c) // bs) for c in suffix) + b      # + one block per append
        nb = prefix // bs + private
        max_blocks = -(-(prefix + 512 + 1) // bs)
        return Workload(name, seed, b, 32, 8, 128, bs, "bf16", "bf16", 1 / math.sqrt(128), 0,
                        ctx, nb, None, max_blocks, append_tokens=b, prefix_len=prefix,
                        alloc_seed=0xC0FFEE)
    if name == "longctx_fp8":
        b, bs, c = 4, bs_x, 131072
        ctx = np.full(b, c, dtype=np.int32)
        nb = b * c // bs
        return Workload(name, seed, b, 64, 8, 128, bs, "fp8_e4m3", "bf16", 1 / math.sqrt(128),
                        512, ctx, nb, _shuffled_tables(seed, ctx, bs, nb, c // bs), c // bs)
    raise KeyError(name)


# -- values -------------------------------------------------------------------

def queries_f32(w):
    """float32 ``[batch, Hq, D]`` query values (before rounding to ``q_dtype``)."""
    n = w.batch * w.n_q_heads * w.head_dim
    return normal_f32(w.seed, _stream(S_Q), n).reshape(w.batch, w.n_q_heads, w.head_dim)


def kv_tokens_f32(w, which, seq, lo, hi):
    """float32 ``[hi-lo, Hkv, D]`` values of logical tokens ``lo..hi-1`` of a sequence.

    ``which`` is "k" or "v".  In the prefix workload tokens below the prefix
    length come from one shared stream, the rest from the sequence's own.
    """
    row = w.n_kv_heads * w.head_dim
    out = np.empty((hi - lo, w.n_kv_heads, w.head_dim), dtype=np.float32)
    if hi <= lo:
        return out
    if w.prefix_len:
        p_hi = min(hi, w.prefix_len)
        if lo < p_hi:
            st = _stream(S_PREFIX_K if which == "k" else S_PREFIX_V)
            out[:p_hi - lo] = normal_f32(w.seed, st, (p_hi - lo) * row, lo * row).reshape(-1, w.n_kv_heads, w.head_dim)
        s_lo = max(lo, w.prefix_len)
        if s_lo < hi:
            st = _stream(S_K if which == "k" else S_V, seq)
            off = (s_lo - w.prefix_len) * row
            out[s_lo - lo:] = normal_f32(w.seed, st, (hi - s_lo) * row, off).reshape(-1, w.n_kv_heads, w.head_dim)
        return out
    st = _stream(S_K if which == "k" else S_V, seq)
    return normal_f32(w.seed, st, (hi - lo) * row, lo * row).reshape(-1, w.n_kv_heads, w.head_dim)


def append_slots(w):
    """int64 slots of the ``gqa_bf16`` 32-token append: distinct unused slots.

    Unused slots are the tail slots of each sequence's last block and every
    slot of the spare blocks (drawn without replacement).
    """
    bs = w.block_size
    used = set()
    for s, c in enumerate(w.context_lens):
        for j in range(-(-int(c) // bs)):
            used.add(int(w.block_tables[s, j]))
    free = []
    for s, c in enumerate(w.context_lens):
        n = -(-int(c) // bs)
        last = int(w.block_tables[s, n - 1])
        free.extend(last * bs + o for o in range(int(c) - (n - 1) * bs, bs))
    for b in range(w.num_blocks):
        if b not in used:
            free.extend(b * bs + o for o in range(bs))
    free = np.array(sorted(free), dtype=np.int64)
    return sample_without_replacement(w.seed, _stream(S_APPEND_SLOTS), free, w.append_tokens)


def append_tokens_f32(w, which):
    """float32 ``[append_tokens, Hkv, D]`` values of the appended tokens (``gqa_bf16``)."""
    st = _stream(S_APPEND_K if which == "k" else S_APPEND_V)
    n = w.append_tokens * w.n_kv_heads * w.head_dim
    return normal_f32(w.seed, st, n).reshape(w.append_tokens, w.n_kv_heads, w.head_dim)


def build_prefix_tables(w, allocator):
    """Block tables of the prefix workload, made by calling ``allocator``.

    ``allocator`` is anything with ``append_slot(row, n, pos, block_size)``
    and ``fork(row, n)`` (the library's or the oracle's).  Sequence 0 writes
    the prefix, every other sequence shares its blocks (fork), then each
    sequence writes its private suffix and the step's new token (position
    ``context_lens[s]``).  Only the order of calls is fixed here; block ids
    and slots are whatever the allocator returns.  Returns ``(tables int32
    [batch, max_blocks], decode context lengths, slots of the new tokens)``.
    """
    bs = w.block_size
    rows = [[-1] * w.max_blocks for _ in range(w.batch)]
    nblk = [0] * w.batch
    for pos in range(w.prefix_len):
        _, nblk[0], _ = allocator.append_slot(rows[0], nblk[0], pos, bs)
    for s in range(1, w.batch):
        allocator.fork(rows[0], nblk[0])
        rows[s][:nblk[0]] = rows[0][:nblk[0]]
        nblk[s] = nblk[0]
    new_slots = []
    for s in range(w.batch):
        for pos in range(w.prefix_len, int(w.context_lens[s]) + 1):
            slot, nblk[s], cow = allocator.append_slot(rows[s], nblk[s], pos, bs)
            if cow is not None:
                raise RuntimeError("the prefix blocks are full: no copy-on-write expected")
        new_slots.append(slot)
    tables = np.array([[max(b, 0) for b in r] for r in rows], dtype=np.int32)
    return tables, w.context_lens.astype(np.int64) + 1, np.array(new_slots, dtype=np.int64)


def fp8_scale_of(values_f32):
    """The per-tensor FP8 scale the workloads use: largest |value| / 448, in float32."""
    return np.float32(np.float32(np.max(np.abs(values_f32))) / np.float32(448.0))


def cast(values_f32, dtype):
    """Round float32 values to the storage of ``dtype`` (f32 / f16 / bf16 bits).

    Input preparation only: bf16 uses torch's round-to-nearest-even cast.
    """
    if dtype == "f32":
        return np.asarray(values_f32, dtype=np.float32)
    if dtype == "f16":
        return np.asarray(values_f32, dtype=np.float32).astype(np.float16)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(values_f32, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)
