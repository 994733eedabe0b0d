"""Parallel sampling end to end on the device: fork, copy-on-write, append,
decode.

dev.to "Why LLMs Run Out of VRAM: KV Cache Fragmentation and How
PagedAttention Fixes It", section 5 "Superpowers of Paged Memory: Zero-Copy
Forking", 1. "Parallel Sampling & Tree Search": the branches of one prompt
share its physical blocks through reference counts; a branch's first write
into a shared block gives it a private copy of that block (copy-on-write);
four branches sharing a prompt hold its memory once instead of four times.

Here a prompt of 40 tokens (two full 16-token blocks and a third holding 8)
is written through the library's allocator and KV append, forked into four
branches, and each branch appends its own token at position 40.  Three of the
four branches find the third block shared and copy it (pa_alloc_append_slot
returns each (source, destination) pair; one pa_copy_blocks call copies them
all before the new tokens are written); the last one is then the block's
only holder and writes in place.  Checked against the oracle:
  - the allocator's state, bit for bit, after every call (oracle/allocator.py
    driven with the same calls);
  - both pools, byte for byte (the oracle's append and a plain block copy);
  - each branch's decode output against the plain attention definition over
    that branch's own logical tokens (prompt + its token), and against the
    oracle's paged decode over the oracle pool;
  - the shared full prompt blocks: held once for four branches (75% less
    prompt memory than four private copies)."""

import math

import numpy as np
import pytest
import torch

import synth
from harness import POISON, TOL, assert_close, to_numpy_storage, to_torch
from oracle import attention as oatt
from oracle import cache as ocache
from oracle import numerics
from oracle.allocator import BlockAllocator as OAlloc
from synth import workloads as wl

pytestmark = pytest.mark.gpu

PROMPT, BRANCHES, BS, HQ, HKV, D = 40, 4, 16, 32, 8, 128


def _same_state(lib_alloc, model):
    free, ref = lib_alloc.dump()
    assert free == list(model.free) and ref == list(model.ref)


@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp8_e4m3", "bf16"), ("f16", "f16"), ("f32", "f32")])
def test_fork_cow_append_decode_matches_oracle(pa, cuda, kv, q):
    src = "f32" if kv == "fp8_e4m3" else kv
    num_blocks, cap, seed = 64, 8, 31
    alloc, model = pa.BlockAllocator(num_blocks, seed), OAlloc(num_blocks, seed)

    # token values: the prompt's, then one new token per branch
    k_prompt = synth.normal_f32(seed, 1, PROMPT * HKV * D).reshape(PROMPT, HKV, D)
    v_prompt = synth.normal_f32(seed, 2, PROMPT * HKV * D).reshape(PROMPT, HKV, D)
    k_new = synth.normal_f32(seed, 3, BRANCHES * HKV * D).reshape(BRANCHES, HKV, D)
    v_new = synth.normal_f32(seed, 4, BRANCHES * HKV * D).reshape(BRANCHES, HKV, D)
    q_store = wl.cast(synth.normal_f32(seed, 5, BRANCHES * HQ * D).reshape(BRANCHES, HQ, D), q)
    k_scale = v_scale = 1.0
    if kv == "fp8_e4m3":
        k_scale = float(wl.fp8_scale_of(np.concatenate([k_prompt.ravel(), k_new.ravel()])))
        v_scale = float(wl.fp8_scale_of(np.concatenate([v_prompt.ravel(), v_new.ravel()])))
    ks_src, vs_src = wl.cast(k_prompt, src), wl.cast(v_prompt, src)
    kn_src, vn_src = wl.cast(k_new, src), wl.cast(v_new, src)
    desc = pa.CacheDesc(num_blocks, BS, HKV, D, kv, k_scale, v_scale)
    kc, vc = desc.new_pools(cuda, fill=POISON)
    kp = ocache.new_pool(num_blocks, HKV, BS, D, kv)
    vp = ocache.new_pool(num_blocks, HKV, BS, D, kv)
    kp.view(np.uint8)[...] = POISON
    vp.view(np.uint8)[...] = POISON

    # the prompt, written through the allocator: slots, then one append call
    row, n, row_m, n_m = [-1] * cap, 0, [-1] * cap, 0
    slots = []
    for pos in range(PROMPT):
        s, n, cow = alloc.append_slot(row, n, pos, BS)
        s_m, n_m, cow_m = model.append_slot(row_m, n_m, pos, BS)
        assert (s, n, cow) == (s_m, n_m, cow_m) and cow is None
        slots.append(s)
    _same_state(alloc, model)
    pa.kv_append(desc, to_torch(ks_src, src, cuda), to_torch(vs_src, src, cuda),
                 torch.tensor(slots, dtype=torch.int64, device=cuda), kc, vc)
    ocache.kv_append(kp, vp, ks_src, vs_src, slots, src, kv, k_scale, v_scale)

    # fork: branches 1..3 share every prompt block with branch 0
    rows = [list(row)]
    for b in range(1, BRANCHES):
        alloc.fork(row, n)
        model.fork(row_m, n_m)
        rows.append(list(row))
    _same_state(alloc, model)
    assert all(alloc.refcount(blk) == BRANCHES for blk in row[:n])

    # each branch's token at position PROMPT: the third block is shared, so
    # the first three branches take private copies; the last writes in place
    new_slots, pairs = [], []
    for b in range(BRANCHES):
        r_m = list(rows[b])
        s, nb, cow = alloc.append_slot(rows[b], n, PROMPT, BS)
        s_m, nb_m, cow_m = model.append_slot(r_m, n, PROMPT, BS)
        assert (s, nb, cow) == (s_m, nb_m, cow_m) and rows[b] == r_m and nb == n
        assert (cow is not None) == (b < BRANCHES - 1)
        if cow is not None:
            assert cow[0] == row[2] and cow[1] not in row
            pairs.append(cow)
        new_slots.append(s)
        _same_state(alloc, model)
    assert len(set(new_slots)) == BRANCHES
    src_ids = torch.tensor([p[0] for p in pairs], dtype=torch.int32, device=cuda)
    dst_ids = torch.tensor([p[1] for p in pairs], dtype=torch.int32, device=cuda)
    pa.copy_blocks(desc, kc, vc, src_ids, dst_ids)          # before the in-place write below (stream order)
    for a, b in pairs:
        kp[b] = kp[a]
        vp[b] = vp[a]
    pa.kv_append(desc, to_torch(kn_src, src, cuda), to_torch(vn_src, src, cuda),
                 torch.tensor(new_slots, dtype=torch.int64, device=cuda), kc, vc)
    ocache.kv_append(kp, vp, kn_src, vn_src, new_slots, src, kv, k_scale, v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(to_numpy_storage(kc, kv).view(np.uint8), kp.view(np.uint8)), "K pool"
    assert np.array_equal(to_numpy_storage(vc, kv).view(np.uint8), vp.view(np.uint8)), "V pool"

    # decode every branch over its own 41 tokens
    tables = np.array(rows, dtype=np.int32)
    ctx = np.full(BRANCHES, PROMPT + 1, dtype=np.int32)
    scale = 1.0 / math.sqrt(D)
    for part in (-1, 16):      # whole context, and one partition per block (fused merge)
        out = pa.decode_attention(desc, to_torch(q_store, q, cuda), kc, vc, torch.from_numpy(tables).to(cuda),
                                  torch.from_numpy(ctx).to(cuda), scale, partition=part)
        got = out.cpu().numpy()
        paged = oatt.decode_attention_paged(q_store, kp, vp, tables, ctx, scale, kv, k_scale, v_scale, q_dtype=q)
        for b in range(BRANCHES):
            logical = []
            for vals, new, sc in ((ks_src, kn_src, k_scale), (vs_src, vn_src, v_scale)):
                toks = np.concatenate([vals, new[b:b + 1]])
                logical.append(numerics.to_f64(numerics.store(toks, src, kv, sc), kv, sc))
            expect = oatt.decode_attention_contiguous(numerics.to_f64(q_store[b], q), logical[0], logical[1], scale)
            assert_close(got[b], expect, TOL[kv], f"{kv} branch {b} partition {part}")
            assert_close(got[b], paged[b], TOL[kv], f"{kv} branch {b} partition {part} (paged oracle)")

    # [DEV] section 5: the full prompt blocks are held once by all four
    # branches; the partly filled one became four private blocks
    n_full = PROMPT // BS
    assert all(alloc.refcount(blk) == BRANCHES for blk in row[:n_full])
    held_full = len({r[j] for r in rows for j in range(n_full)})
    assert 1 - held_full / (BRANCHES * n_full) == 0.75
    held = len({blk for r in rows for blk in r[:n]})
    assert held == n_full + BRANCHES
    assert alloc.free_count == num_blocks - held
