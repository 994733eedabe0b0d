"""GPU parity of decode over slid windows (pa_decode_attention_window) and of
the allocator's truncate driving it.

[VK] "PagedAttention: the idea" / "A minimal PyTorch sketch" (truncate): the
oldest whole pages go back to the allocator and the rest of the drop is an
offset into the first kept page.  Each sequence attends the positions
[start, ctx) of its row; table entries of blocks wholly before a start are
set to -1 here, so a read of one would raise PA_DEVFLAG_BLOCK_RANGE."""

import numpy as np
import pytest
import torch

import synth
from harness import POISON, TOL, Case, assert_close, to_torch
from oracle import attention as oatt
from oracle import numerics
from synth import workloads

pytestmark = pytest.mark.gpu


def _window_case(case, starts):
    """Tables with the entries before each start released (-1)."""
    tables = case.tables.copy()
    for s, st in enumerate(starts):
        st = max(0, min(int(st), int(case.ctx[s])))
        tables[s, :st // case.bs] = -1
    return tables


def _run(pa, cuda, case, starts, partition, out_dtype="f32"):
    kc, vc = case.gpu_pools(pa, cuda)
    tables = _window_case(case, starts)
    status = pa.new_status(cuda)
    q = to_torch(case.q_store, case.q_dtype, cuda)
    out = pa.decode_attention(case.desc(pa), q, kc, vc, torch.from_numpy(tables).to(cuda),
                              torch.from_numpy(case.ctx).to(cuda), case.scale, partition=partition,
                              out_dtype=out_dtype, status=status,
                              context_starts=torch.tensor(np.asarray(starts, np.int32), device=cuda))
    torch.cuda.synchronize()
    kp, vp = case.oracle_pools()
    want = oatt.decode_attention_paged(case.q_store, kp, vp, tables, case.ctx, case.scale, case.kv_dtype,
                                       case.k_scale, case.v_scale, q_dtype=case.q_dtype,
                                       context_starts=np.clip(starts, 0, case.ctx))
    return out, want, pa.read_device_status(status)


@pytest.mark.parametrize("kv,q,bs,partition", [
    ("bf16", "bf16", 16, 0), ("bf16", "bf16", 16, 256), ("bf16", "bf16", 16, 32), ("bf16", "bf16", 16, -1),
    ("f16", "f16", 8, 64), ("bf16", "bf16", 32, 128), ("fp8_e4m3", "bf16", 16, 512), ("fp8_e4m3", "bf16", 8, 32),
    ("f32", "f32", 16, 64)])
@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_window_matches_oracle(pa, cuda, kernel, kv, q, bs, partition):
    ctx = [3000, 700, 129, 40, 16, 5, 77]
    # starts: deep into the context, none, at a chunk edge, one short of the
    # end, a whole first block, an empty window, and a start in the second
    # half of a 16-token chunk (8-token blocks: the chunk's first block is released)
    starts = [1234, 0, 128, 39, 16, 5, 29]
    case = Case(batch=7, hq=16, hkv=4, d=128, bs=bs, kv_dtype=kv, q_dtype=q, ctx=ctx, seed=61)
    out, want, flags = _run(pa, cuda, case, starts, partition)
    assert flags == 0, f"device status {flags:#x}: a block before a window start was read"
    got = out.cpu().numpy()
    assert_close(got, want, TOL[kv], f"window {kv} bs{bs} P{partition}")
    assert np.all(got[5] == 0)          # empty window


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3"])
def test_window_starts_out_of_range_are_clamped_and_flagged(pa, cuda, kv):
    case = Case(batch=3, hq=8, hkv=1, d=128, bs=16, kv_dtype=kv, q_dtype="bf16", ctx=[100, 50, 33], seed=62)
    kc, vc = case.gpu_pools(pa, cuda)
    status = pa.new_status(cuda)
    q = to_torch(case.q_store, case.q_dtype, cuda)
    starts = torch.tensor([-5, 60, 10], dtype=torch.int32, device=cuda)       # below 0, beyond ctx, fine
    out = pa.decode_attention(case.desc(pa), q, kc, vc, torch.from_numpy(case.tables).to(cuda),
                              torch.from_numpy(case.ctx).to(cuda), case.scale, status=status,
                              context_starts=starts)
    torch.cuda.synchronize()
    assert pa.read_device_status(status) & 4          # PA_DEVFLAG_CONTEXT_RANGE
    kp, vp = case.oracle_pools()
    want = oatt.decode_attention_paged(case.q_store, kp, vp, case.tables, case.ctx, case.scale, case.kv_dtype,
                                       case.k_scale, case.v_scale, q_dtype=case.q_dtype,
                                       context_starts=[0, 50, 10])
    got = out.cpu().numpy()
    assert_close(got, want, TOL[kv], "clamped starts")
    assert np.all(got[1] == 0)


def test_truncate_then_reuse_released_blocks(pa, cuda):
    """Sequences written through the library's allocator, windows slid with
    pa_alloc_truncate, the released blocks handed to a new sequence and
    overwritten: decode over the windows still equals attention over each
    sequence's last `keep` tokens, computed on the unpaged data."""
    bs, hkv, hq, d = 16, 2, 8, 128
    n_tok, keeps = [300, 157, 64], [100, 150, 17]
    nb = 64
    alloc = pa.BlockAllocator(nb, 11)
    desc = pa.CacheDesc(nb, bs, hkv, d, "bf16", 1.0, 1.0)
    kc, vc = desc.new_pools(cuda, fill=POISON)
    rows, nblk, kv_src = [], [], []
    for s, n in enumerate(n_tok):
        k = workloads.cast(synth.normal_f32(70, (1 << 32) | s, n * hkv * d).reshape(n, hkv, d), "bf16")
        v = workloads.cast(synth.normal_f32(70, (2 << 32) | s, n * hkv * d).reshape(n, hkv, d), "bf16")
        row, nb_s, slots = [-1] * 24, 0, []
        for t in range(n):
            slot, nb_s, _ = alloc.append_slot(row, nb_s, t, bs)
            slots.append(slot)
        pa.kv_append(desc, to_torch(k, "bf16", cuda), to_torch(v, "bf16", cuda),
                     torch.tensor(slots, dtype=torch.int64, device=cuda), kc, vc)
        rows.append(row), nblk.append(nb_s), kv_src.append((k, v))
    starts, lens = [], []
    for s in range(3):
        nblk[s], st, ln = alloc.truncate(rows[s], nblk[s], 0, n_tok[s], keeps[s], bs)
        starts.append(st), lens.append(ln)
    # a new sequence takes the released blocks and overwrites them with other values
    junk_row, junk_n, junk_slots = [-1] * nb, 0, []
    for t in range(alloc.free_count * bs):
        slot, junk_n, _ = alloc.append_slot(junk_row, junk_n, t, bs)
        junk_slots.append(slot)
    junk = torch.full((len(junk_slots), hkv, d), 1000.0, dtype=torch.bfloat16, device=cuda)
    pa.kv_append(desc, junk, junk, torch.tensor(junk_slots, dtype=torch.int64, device=cuda), kc, vc)
    q_store = workloads.cast(synth.normal_f32(70, 9, 3 * hq * d).reshape(3, hq, d), "bf16")
    status = pa.new_status(cuda)
    out = pa.decode_attention(desc, to_torch(q_store, "bf16", cuda), kc, vc,
                              torch.tensor(np.array(rows, np.int32)[:, :24], device=cuda),
                              torch.tensor(lens, dtype=torch.int32, device=cuda), 1 / np.sqrt(d), status=status,
                              context_starts=torch.tensor(starts, dtype=torch.int32, device=cuda))
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0
    qf = numerics.to_f64(q_store, "bf16")
    for s in range(3):
        k, v = kv_src[s]
        K = numerics.to_f64(k[n_tok[s] - keeps[s]:], "bf16")
        V = numerics.to_f64(v[n_tok[s] - keeps[s]:], "bf16")
        want = oatt.decode_attention_contiguous(qf[s], K, V, 1 / np.sqrt(d))
        assert_close(out[s].cpu().numpy(), want, TOL["bf16"], f"sequence {s}")
