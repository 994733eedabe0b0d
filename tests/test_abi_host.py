"""The C-ABI library on the host (no GPU needed): every declared symbol is
exported, and the host-side entry points match the oracle bit for bit."""

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import cache as ocache
from oracle import closed_forms
from oracle.allocator import AllocError as OAllocError
from oracle.allocator import BlockAllocator as OAlloc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "pagedattn.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(built_lib):
    names = _declared()
    assert len(names) >= 20
    lib = ctypes.CDLL(built_lib)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_declares_every_symbol(pa):
    from paged_kv_cache_257_gb300 import _native
    assert set(_declared()) == set(_native.SIGNATURES)


def test_decode_deterministic_setting_round_trips(pa):
    prev = pa.decode_deterministic()
    try:
        assert pa.set_decode_deterministic(True) == prev
        assert pa.decode_deterministic() is True
        assert pa.set_decode_deterministic(False) is True
        assert pa.decode_deterministic() is False
    finally:
        pa.set_decode_deterministic(prev)


def test_decode_kernel_setting_round_trips_and_rejects_unknown_values(pa):
    from paged_kv_cache_257_gb300 import _native
    lib = _native.lib()
    prev = pa.decode_kernel()
    try:
        assert pa.set_decode_kernel("warp") == prev
        assert pa.decode_kernel() == "warp" and lib.pa_get_decode_kernel() == 2
        assert pa.set_decode_kernel("cta") == "warp"
        assert lib.pa_set_decode_kernel(7) == 1                  # PA_ERR_INVALID, setting unchanged
        assert lib.pa_set_decode_kernel(-1) == 1
        assert pa.decode_kernel() == "cta"
        assert pa.set_decode_kernel("auto") == "cta"
    finally:
        pa.set_decode_kernel(prev)


def test_version_and_status_strings(pa):
    from paged_kv_cache_257_gb300 import _native
    assert "sm_103a" in pa.version()
    lib = _native.lib()
    for code, name in _native.STATUS.items():
        assert lib.pa_status_string(code).decode() == name


@pytest.mark.parametrize("layers,hkv,d,dtype", [(40, 40, 128, "f16"), (32, 8, 128, "bf16"), (80, 8, 128, "fp8_e4m3"),
                                                (1, 2, 64, "f32")])
def test_kv_bytes_per_token_matches_closed_form(pa, layers, hkv, d, dtype):
    b = closed_forms.DTYPE_BYTES[dtype]
    assert pa.kv_bytes_per_token(layers, hkv, d, dtype) == closed_forms.kv_bytes_per_token(layers, hkv, d, b)
    assert pa.dtype_size(dtype) == b


def test_slot_mapping_matches_oracle(pa):
    rng = np.random.default_rng(0)
    for bs in (8, 16, 32):
        tables = rng.permutation(4000)[:40 * 20].reshape(20, 40).astype(np.int32)
        seq = rng.integers(0, 20, 500).astype(np.int32)
        pos = rng.integers(0, 40 * bs, 500).astype(np.int32)
        got = pa.compute_slot_mapping(tables, seq, pos, bs)
        assert np.array_equal(got, ocache.slot_mapping(tables, seq, pos, bs))


def test_slot_mapping_rejects_bad_positions(pa):
    tables = np.zeros((2, 3), dtype=np.int32)
    for seq, pos in ((0, 48), (0, -1), (2, 0)):
        with pytest.raises(pa.NativeError) as e:
            pa.compute_slot_mapping(tables, [seq], [pos], 16)
        assert e.value.status == "PA_ERR_RANGE"


# ------------------------------------------------------------- allocator

def _same(lib_alloc, model):
    assert lib_alloc.dump() == model.dump()
    assert lib_alloc.free_count == model.free_count


@pytest.mark.parametrize("seed", [0, 1, 42, 0xC0FFEE])
def test_allocator_handout_order(pa, seed):
    a, m = pa.BlockAllocator(300, seed), OAlloc(300, seed)
    _same(a, m)
    assert [a.alloc() for _ in range(300)] == [m.alloc() for _ in range(300)]
    _same(a, m)


def _apply(obj, op, *args):
    try:
        return ("ok", getattr(obj, op)(*args))
    except (OAllocError,) as e:
        return ("err", e.status)
    except Exception as e:  # library AllocError
        if hasattr(e, "status"):
            return ("err", e.status)
        raise


def test_allocator_random_trace_is_bit_exact(pa):
    rng = np.random.default_rng(1)
    a, m = pa.BlockAllocator(96, 7), OAlloc(96, 7)
    rows_a, rows_m, nblk = [], [], []
    for step in range(4000):
        op = rng.integers(0, 6)
        if op == 0 or not rows_a:                         # start a sequence
            rows_a.append([-1] * 8)
            rows_m.append([-1] * 8)
            nblk.append(0)
            continue
        i = int(rng.integers(len(rows_a)))
        if op in (1, 2):                                  # append a token at the end
            pos = int(rng.integers(0, nblk[i] * 16 + 1))
            ra = _apply(a, "append_slot", rows_a[i], nblk[i], pos, 16)
            rm = _apply(m, "append_slot", rows_m[i], nblk[i], pos, 16)
            assert ra == rm
            assert rows_a[i] == rows_m[i]
            if ra[0] == "ok":
                nblk[i] = ra[1][1]
        elif op == 3:                                     # fork
            ra = _apply(a, "fork", rows_a[i], nblk[i])
            rm = _apply(m, "fork", rows_m[i], nblk[i])
            assert ra == rm
            if ra[0] == "ok":
                rows_a.append(list(rows_a[i]))
                rows_m.append(list(rows_m[i]))
                nblk.append(nblk[i])
        elif op == 4:                                     # finish a sequence
            ra = _apply(a, "free_sequence", rows_a[i], nblk[i])
            rm = _apply(m, "free_sequence", rows_m[i], nblk[i])
            assert ra == rm
            rows_a.pop(i), rows_m.pop(i), nblk.pop(i)
        else:                                             # raw single-block calls, some invalid
            b = int(rng.integers(-2, 100))
            fn = ("incref", "decref", "cow")[int(rng.integers(3))]
            assert _apply(a, fn, b) == _apply(m, fn, b)
        _same(a, m)


def test_allocator_cow_scenario_matches_model(pa):
    for alloc in (pa.BlockAllocator(10), OAlloc(10)):
        row, n = [-1] * 4, 0
        for pos in range(20):
            _, n, _ = alloc.append_slot(row, n, pos, 16)
        alloc.fork(row, n)
        child = list(row)
        slot, _, cow = alloc.append_slot(child, n, 20, 16)
        assert cow == (1, 2) and slot == 2 * 16 + 4


def test_allocator_errors(pa):
    a = pa.BlockAllocator(1)
    a.alloc()
    with pytest.raises(pa.AllocError) as e:
        a.alloc()
    assert e.value.status == "OOM"
    with pytest.raises(pa.AllocError) as e:
        a.incref(5)
    assert e.value.status == "RANGE"
    with pytest.raises(pa.AllocError):
        pa.BlockAllocator(0)


# ------------------------------------------------- host-side validation

def _call_decode(pa, desc, **over):
    from paged_kv_cache_257_gb300 import _native
    lib = _native.lib()
    args = dict(q=8192, q_dtype=2, hq=32, k=8192, v=8192, bt=8192, max_blocks=256, ctx=8192, batch=4,
                scale=0.088, part=0, ws=None, ws_bytes=0, out=8192, out_dtype=0)
    args.update(over)
    c = desc.c()
    return lib.pa_decode_attention(ctypes.byref(c), args["q"], args["q_dtype"], args["hq"], args["k"], args["v"],
                                   args["bt"], args["max_blocks"], args["ctx"], args["batch"], args["scale"],
                                   args["part"], args["ws"], args["ws_bytes"], args["out"], args["out_dtype"],
                                   None, None)


def test_decode_rejects_bad_arguments_before_any_launch(pa):
    d = pa.CacheDesc(1024, 16, 8, 128, "bf16")
    assert _call_decode(pa, d, q=None) == 1
    assert _call_decode(pa, d, hq=30) == 1                       # not a multiple of Hkv
    assert _call_decode(pa, d, q=8194) == 1                      # misaligned
    assert _call_decode(pa, d, part=24) == 1                     # not a multiple of 16
    assert _call_decode(pa, d, ws=None, ws_bytes=0) == 1         # split needs a workspace
    assert _call_decode(pa, d, out_dtype=3) == 4                 # FP8 output unsupported
    assert _call_decode(pa, d, scale=float("inf")) == 1
    assert _call_decode(pa, d, batch=0) == 0                     # empty batch: no-op
    assert _call_decode(pa, pa.CacheDesc(1024, 16, 8, 96, "bf16")) == 4
    assert _call_decode(pa, pa.CacheDesc(1024, 12, 8, 128, "bf16")) == 4
    assert _call_decode(pa, pa.CacheDesc(1024, 16, 8, 128, "fp8_e4m3", 0.0, 1.0)) == 1


def test_decode_rejects_grids_beyond_the_launch_limits(pa):
    """Limits checked before any launch: 65535 sequences (the grid's z
    extent), 32768 partitions per sequence, and tables of 2^31 tokens."""
    d = pa.CacheDesc(1024, 16, 8, 128, "bf16")
    assert _call_decode(pa, d, batch=65536, part=-1) == 4
    assert _call_decode(pa, d, max_blocks=32769, part=16, ws=8192, ws_bytes=1 << 40) == 4   # 32769 partitions
    assert _call_decode(pa, d, max_blocks=1 << 27, part=-1) == 4                          # 2^31 tokens
    assert pa.partition_size(d, 4, 32, 1 << 27, -1) == -1


def test_noalloc_rejects_null_pointers_and_oversized_problems_on_the_host(pa):
    """The allocation-free entry point answers before any CUDA call: a null
    input or output of a split call is PA_ERR_INVALID, a workspace beyond
    its array PA_ERR_RANGE."""
    from paged_kv_cache_257_gb300 import _native
    lib = _native.lib()
    c = pa.CacheDesc(1024, 16, 8, 128, "bf16").c()
    assert pa.decode_workspace_size(pa.CacheDesc(1024, 16, 8, 128, "bf16"), 2, 32, 64, 256) > 0

    def call(**o):
        a = dict(q=4096, kc=4096, vc=4096, bt=4096, cl=4096, out=4096, part=256, batch=2, mb=64)
        a.update(o)
        return lib.pa_decode_attention_noalloc(ctypes.byref(c), a["q"], 2, 32, a["kc"], a["vc"], a["bt"], a["mb"],
                                               a["cl"], a["batch"], 0.088, a["part"], a["out"], 0, None, None)
    for name in ("q", "kc", "vc", "bt", "cl", "out"):
        assert call(**{name: None}) == 1, name
    big = pa.CacheDesc(32768, 16, 8, 128, "fp8_e4m3", 0.01, 0.01)
    assert pa.decode_workspace_size(big, 4, 64, 8192, 512) > _native.NOALLOC_SCRATCH_BYTES
    cb = big.c()
    assert lib.pa_decode_attention_noalloc(ctypes.byref(cb), 4096, 2, 64, 4096, 4096, 4096, 8192, 4096, 4, 0.088,
                                           512, 4096, 0, None, None) == 3


def test_append_rejects_bad_arguments(pa):
    from paged_kv_cache_257_gb300 import _native
    lib = _native.lib()
    c = pa.CacheDesc(64, 16, 2, 64, "bf16").c()
    ok = dict(k=4096, v=4096, src=2, slots=4096, n=3, kc=4096, vc=4096)

    def call(**o):
        a = dict(ok)
        a.update(o)
        return lib.pa_kv_append(ctypes.byref(c), a["k"], a["v"], a["src"], a["slots"], a["n"], a["kc"], a["vc"],
                                None, None)
    assert call(n=0) == 0
    assert call(k=None) == 1
    assert call(src=1) == 4               # f16 source into a bf16 cache
    assert call(slots=4100) == 1          # int64 slots misaligned
    assert call(n=-1) == 1


def test_workspace_and_partition_sizes(pa):
    d = pa.CacheDesc(32768, 16, 8, 128, "fp8_e4m3", 0.01, 0.01)
    assert pa.partition_size(d, 4, 64, 8192, 512) == 512
    # merge tickets (4 x 8 groups, padded to 256 B), partial outputs, partial (max, sum)
    assert pa.decode_workspace_size(d, 4, 64, 8192, 512) == 256 + 4 * 64 * 256 * 128 * 4 + 4 * 64 * 256 * 2 * 4
    assert pa.partition_size(d, 4, 64, 8192, -1) == 131072
    assert pa.decode_workspace_size(d, 4, 64, 8192, -1) == 0         # no split, no workspace
    assert pa.partition_size(d, 4, 64, 8192, 100) == -1
    auto = pa.partition_size(d, 4, 64, 8192, 0)
    assert auto > 0 and auto % 16 == 0


def test_plan_partition_follows_the_wave_model(pa):
    """Costs worked by hand: waves = ceil(items / (5 x 152)), each as long as
    its longest item plus 192 tokens; ties keep the larger partition."""
    gqa = pa.CacheDesc(8192, 16, 8, 128, "bf16", 1.0, 1.0)
    # 32 full 4096-token sequences, 8 KV heads: 4096 -> 1 x 4288, 2048 -> 1 x 2240,
    # 1024 -> 2 x 1216, 512 -> 3 x 704 = 2112 (least), 256 -> 6 x 448
    assert pa.plan_partition(gqa, 32, 32, 256, [4096] * 32, 152) == 512
    # the same batch at 1024 tokens each: 512 -> 1 x 704 beats 256 -> 2 x 448 and the whole 1 x 1216
    assert pa.plan_partition(gqa, 32, 32, 256, [1024] * 32, 152) == 512
    # one short sequence: every candidate costs 100 + 192; the whole context wins the tie
    assert pa.plan_partition(gqa, 1, 32, 256, [100], 152) == 4096
    # unknown lengths are taken as full
    assert pa.plan_partition(gqa, 32, 32, 256, None, 152) == 512
    fp8 = pa.CacheDesc(32768, 16, 8, 128, "fp8_e4m3", 0.01, 0.01)
    # 4 x 131072 tokens, 64 query heads (one group of 8 per KV head): 2048 -> 3 x 2240
    # beats 1024 -> 6 x 1216, 512 -> 11 x 704 and 4096 -> 2 x 4288; the finer grid's
    # 2816 (47 x 32 = 1504 items, 2 x (2800 + 192) = 5984) spans two waves and is not taken
    assert pa.plan_partition(fp8, 4, 64, 8192, [131072] * 4, 152) == 2048
    # a batch of long items that leaves a third of the CTA slots idle when whole:
    # 64 sequences of 2049..2561 tokens (8 KV heads, whole = 2576): 512 items,
    # 1 x (2561 + 192); at 2304 the 32 longest split in two (their shares <= 1296):
    # (32 + 2 x 32) x 8 = 768 > 760 slots, 2 waves; at 2432 the 16 longest split:
    # 640 items, 1 x (2432 + 192) = 2624, the least
    lens = [2049 + (512 * i) // 63 for i in range(64)]
    assert pa.plan_partition(gqa, 64, 32, 161, lens, 152) == 2432
    # a ragged batch plans from its real lengths: one long sequence among short
    # ones is cut finest, as all its pieces still fit one wave:
    # 256 -> (16 + 31 x 2) x 8 = 624 items, 1 x (256 + 192) beats 512 -> 1 x 704
    assert pa.plan_partition(gqa, 32, 32, 256, [4096] + [300] * 31, 152) == 256
    # ... and a long batch takes the finer grid when it fills one wave: 31 x 4096 + 300
    # at 1920 -> 3 shares of 1376 each, (31 x 3 + 1) x 8 = 752 items, 1 x (1376 + 192) =
    # 1568, beats 512 -> 1992 items, 3 x 704 = 2112 (32 x 4096 at 1920 needs 768 items,
    # two waves: 3136, so the full case above keeps 512)
    assert pa.plan_partition(gqa, 32, 32, 256, [4096] * 31 + [300], 152) == 1920
    bs32 = pa.CacheDesc(4096, 32, 8, 128, "bf16", 1.0, 1.0)
    assert pa.plan_partition(bs32, 32, 32, 128, [4096] * 32, 152) % 32 == 0


def test_plan_partition_rejects_bad_arguments(pa):
    d = pa.CacheDesc(8192, 16, 8, 128, "bf16", 1.0, 1.0)
    with pytest.raises(ValueError):
        pa.plan_partition(d, 4, 32, 256, [1, 2, 3], 152)     # 3 lengths for 4 sequences
    with pytest.raises(ValueError):
        pa.plan_partition(d, 4, 30, 256, [1] * 4, 152)       # 30 query heads over 8 KV heads
    # partition_size's automatic choice is the plan for full sequences on this device
    assert pa.partition_size(d, 4, 32, 256, 0) == pa.plan_partition(d, 4, 32, 256, None, 0)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_allocator_truncate_trace_is_bit_exact(pa, bs):
    """Appends at each sequence's end, window slides (some with bad
    arguments), forks and frees: the library and the model agree on every
    result, row and state dump."""
    rng = np.random.default_rng(40 + bs)
    a, m = pa.BlockAllocator(80, 3), OAlloc(80, 3)
    seqs = []   # [row_a, row_m, nblk, start, length]
    for step in range(3000):
        op = rng.integers(0, 8)
        if op == 0 or not seqs:
            seqs.append([[-1] * 12, [-1] * 12, 0, 0, 0])
            continue
        i = int(rng.integers(len(seqs)))
        sq = seqs[i]
        if op in (1, 2, 3):                               # append the next token
            ra = _apply(a, "append_slot", sq[0], sq[2], sq[4], bs)
            rm = _apply(m, "append_slot", sq[1], sq[2], sq[4], bs)
            assert ra == rm and sq[0] == sq[1]
            if ra[0] == "ok":
                sq[2], sq[4] = ra[1][1], sq[4] + 1
        elif op == 4:                                     # slide the window
            keep = int(rng.integers(-1, 3 * bs))
            start = sq[3] if rng.integers(0, 10) else sq[4] + 1      # now and then an inconsistent start
            ra = _apply(a, "truncate", sq[0], sq[2], start, sq[4], keep, bs)
            rm = _apply(m, "truncate", sq[1], sq[2], start, sq[4], keep, bs)
            assert ra == rm and sq[0] == sq[1]
            if ra[0] == "ok":
                sq[2], sq[3], sq[4] = ra[1]
        elif op == 5:                                     # fork
            ra = _apply(a, "fork", sq[0], sq[2])
            assert ra == _apply(m, "fork", sq[1], sq[2])
            if ra[0] == "ok":
                seqs.append([list(sq[0]), list(sq[1]), sq[2], sq[3], sq[4]])
        else:                                             # finish
            ra = _apply(a, "free_sequence", sq[0], sq[2])
            assert ra == _apply(m, "free_sequence", sq[1], sq[2])
            seqs.pop(i)
        _same(a, m)


def test_prefix_block_key_matches_the_oracle(pa):
    from oracle import prefix_cache as opc
    rng = np.random.default_rng(8)
    for n in (0, 1, 8, 16, 32):
        toks = rng.integers(-2**31, 2**31 - 1, n, dtype=np.int64).astype(np.int32)
        parent = int(rng.integers(0, 2**63)) * 2 + 1
        assert pa.PrefixCache.block_key(parent, toks) == opc.block_key(parent, [int(t) for t in toks])


@pytest.mark.parametrize("bs", [8, 16])
def test_prefix_cache_trace_is_bit_exact(pa, bs):
    """Requests drawn from a few shared prompts: match, prefill the rest,
    insert, finish or keep; evictions when the pool runs low.  The library
    and the model agree on every result, row, cache size and allocator dump."""
    from oracle import prefix_cache as opc
    rng = np.random.default_rng(60 + bs)
    nb = 96
    la, lm = pa.BlockAllocator(nb, 4), OAlloc(nb, 4)
    ca, cm = pa.PrefixCache(la, bs), opc.PrefixCache(lm, bs)
    prompts = [list(map(int, rng.integers(0, 30, 80))) for _ in range(3)]
    live = []   # (row_a, row_m, nblk)
    for step in range(600):
        op = rng.integers(0, 10)
        if op < 5:                                          # a new request
            p = prompts[rng.integers(0, 3)]
            toks = p[:int(rng.integers(0, 81))] + list(map(int, rng.integers(0, 30, int(rng.integers(0, 40)))))
            ra, rm = [-1] * 16, [-1] * 16
            ma, mm = ca.match(toks, ra), cm.match(toks, rm)
            assert ma == mm and ra == rm
            n, ok = ma, True
            for t in range(ma * bs, min(len(toks), 16 * bs)):
                xa = _apply(la, "append_slot", ra, n, t, bs)
                xm = _apply(lm, "append_slot", rm, n, t, bs)
                assert xa == xm and ra == rm
                if xa[0] != "ok":
                    ok = False
                    break
                n = xa[1][1]
            if ok:
                ia = _apply(ca, "insert", toks, ra, n)
                assert ia == _apply(cm, "insert", toks, rm, n)
            live.append((ra, rm, n))
        elif op < 8 and live:                               # a request finishes
            ra, rm, n = live.pop(int(rng.integers(len(live))))
            assert _apply(la, "free_sequence", ra, n) == _apply(lm, "free_sequence", rm, n)
        else:                                               # make room
            k = int(rng.integers(0, 12))
            assert ca.evict(k) == cm.evict(k)
        assert ca.size == cm.size
        _same(la, lm)
    ca.destroy(), cm.destroy()
    _same(la, lm)


def test_prefix_cache_insert_errors(pa):
    al = pa.BlockAllocator(8)
    c = pa.PrefixCache(al, 4)
    with pytest.raises(pa.AllocError) as e:
        c.insert(list(range(8)), [0, 1], 2)        # free blocks
    assert e.value.status == "INVALID" and c.size == 0 and al.free_count == 8
    with pytest.raises(pa.AllocError) as e:
        c.insert(list(range(4)), [99], 1)
    assert e.value.status == "RANGE"
