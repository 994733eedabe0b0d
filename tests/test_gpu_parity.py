"""GPU parity: the library (CUDA kernels through the C ABI) against the oracle on
the same seeded inputs.  Pools must match bit for bit after the append;
attention outputs within the tolerance of the cache type:
1e-5 (float32 cache), 1e-2 (16-bit cache), 3e-2 (FP8 cache, oracle on the same
dequantised values), with float32 outputs."""

import math

import numpy as np
import pytest
import torch

from harness import POISON, TOL, Case, assert_close, to_numpy_storage, to_torch
from oracle import numerics

pytestmark = pytest.mark.gpu

RAGGED = [1, 15, 16, 17, 100, 257, 600, 1023]


def _run(pa, cuda, case, partition=None, out_dtype="f32"):
    status = pa.new_status(cuda)
    kc, vc = case.gpu_pools(pa, cuda, status)
    kp, vp = case.oracle_pools()
    assert np.array_equal(to_numpy_storage(kc, case.kv_dtype).view(np.uint8), kp.view(np.uint8)), "K pool"
    assert np.array_equal(to_numpy_storage(vc, case.kv_dtype).view(np.uint8), vp.view(np.uint8)), "V pool"
    out = case.gpu_decode(pa, cuda, kc, vc, out_dtype=out_dtype, partition=partition, status=status)
    assert pa.read_device_status(status) == 0
    expect = case.oracle_out(kp, vp)
    got = out.float().cpu().numpy()
    return got, expect


def test_tiny_workload(pa, cuda):
    from synth import workloads
    w = workloads.make("tiny")
    case = Case(batch=4, hq=4, hkv=2, d=64, bs=16, kv_dtype="f32", q_dtype="f32", ctx=w.context_lens, seed=0)
    got, expect = _run(pa, cuda, case)
    assert_close(got, expect, TOL["f32"], "tiny")


@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("f16", "f16"), ("fp8_e4m3", "bf16"), ("fp8_e4m3", "f16")])
@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (16, 2), (4, 2), (32, 2)])
@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_tensor_core_path_ragged(pa, cuda, kernel, kv, q, hq, hkv):
    case = Case(batch=len(RAGGED), hq=hq, hkv=hkv, d=128, bs=16, kv_dtype=kv, q_dtype=q, ctx=RAGGED, seed=hq + hkv)
    got, expect = _run(pa, cuda, case)
    assert_close(got, expect, TOL[kv], f"{kv} G={hq // hkv} {kernel}")


@pytest.mark.parametrize("hq,hkv", [(6, 2), (10, 2), (24, 2), (32, 1), (64, 1)])
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp8_e4m3", "f16")])
@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_group_sizes_beyond_one_cta(pa, cuda, kernel, kv, q, hq, hkv):
    """G = 3, 5, 12, 32, 64: groups of fewer than 8 heads, and groups split
    over several 8-head work items (12 = 8 + 4)."""
    case = Case(batch=4, hq=hq, hkv=hkv, d=128, bs=16, kv_dtype=kv, q_dtype=q, ctx=[1, 300, 1000, 77], seed=hq)
    got, expect = _run(pa, cuda, case, partition=256)
    assert_close(got, expect, TOL[kv], f"{kv} G={hq // hkv} {kernel}")


@pytest.mark.parametrize("scale", [0.0, 1e-3, 1.0, 30.0])
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp8_e4m3", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_softmax_scale_extremes(pa, cuda, kernel, kv, q, scale):
    """Scale 0 (every token weighs the same: the mean of V), a tiny scale,
    and large ones, where the scores of one chunk jump far past the running
    maximum (the rescale path) and the weights approach one-hot."""
    case = Case(batch=3, hq=8, hkv=2, d=128, bs=16, kv_dtype=kv, q_dtype=q, ctx=[700, 33, 2000], seed=23)
    case.scale = scale
    got, expect = _run(pa, cuda, case, partition=256)
    # float32 caches: the scores' float32 rounding grows with the scale
    # (about |q||k| x 2^-24 per dot product, times the scale, becomes the
    # weights' relative error); the 1e-5 bar holds at 1/sqrt(D) ~ 0.088.
    tol = TOL[kv] * max(1.0, scale * math.sqrt(128)) if kv == "f32" else TOL[kv]
    assert_close(got, expect, tol, f"{kv} scale={scale} {kernel}")
    if scale == 0.0:   # the plain mean of the dequantised values
        kp, vp = case.oracle_pools()
        from oracle import cache as ocache
        v = numerics.to_f64(ocache.gather_logical(vp, case.tables[1], 33, 0), kv, case.v_scale)
        np.testing.assert_allclose(expect[1, 0], v[:, 0].mean(axis=0), rtol=0, atol=1e-12)


@pytest.mark.parametrize("partition", [-1, 16, 64, 256, 512, 0])
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp8_e4m3", "bf16"), ("f32", "f32")])
@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_partition_invariance(pa, cuda, kernel, partition, kv, q):
    case = Case(batch=5, hq=8, hkv=2, d=128, bs=16, kv_dtype=kv, q_dtype=q, ctx=[3000, 1, 511, 512, 513], seed=7)
    got, expect = _run(pa, cuda, case, partition=partition)
    assert_close(got, expect, TOL[kv], f"P={partition} {kernel}")


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("kv,q", [("bf16", "bf16"), ("fp8_e4m3", "bf16"), ("f16", "f32"), ("f32", "f32")])
@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_block_sizes(pa, cuda, kernel, bs, kv, q):
    case = Case(batch=6, hq=8, hkv=4, d=128, bs=bs, kv_dtype=kv, q_dtype=q, ctx=[1, 7, 8, 9, 31, 700], seed=bs)
    got, expect = _run(pa, cuda, case, partition=64)
    assert_close(got, expect, TOL[kv], f"bs={bs} {kernel}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("kv,q", [("f32", "f32"), ("bf16", "f32"), ("fp8_e4m3", "f32"), ("f16", "bf16")])
def test_cuda_core_path(pa, cuda, d, kv, q):
    case = Case(batch=4, hq=6, hkv=2, d=d, bs=16, kv_dtype=kv, q_dtype=q, ctx=[1, 33, 130, 300], seed=d)
    got, expect = _run(pa, cuda, case, partition=128)
    assert_close(got, expect, TOL[kv], f"simt D={d}")


@pytest.mark.parametrize("out_dtype", ["bf16", "f16"])
def test_16bit_outputs_round_the_result(pa, cuda, out_dtype):
    case = Case(batch=3, hq=16, hkv=4, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[1, 40, 900], seed=3)
    got, expect = _run(pa, cuda, case, out_dtype=out_dtype)
    ulp = np.spacing(np.abs(expect).astype(np.float16 if out_dtype == "f16" else np.float32))
    if out_dtype == "bf16":
        ulp = np.maximum(np.abs(expect), 2.0 ** -126) * 2.0 ** -7
    assert np.all(np.abs(got - expect) <= TOL["bf16"] + ulp)


def test_empty_and_single_token_sequences(pa, cuda):
    case = Case(batch=4, hq=8, hkv=8, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[0, 1, 0, 2], seed=11)
    got, expect = _run(pa, cuda, case, partition=-1)
    assert np.array_equal(got[0], np.zeros_like(got[0])) and np.array_equal(got[2], np.zeros_like(got[2]))
    # a single token's output is its value row, dequantised (within float32 rounding)
    v1 = numerics.to_f64(case.v_src[1][0], "bf16")
    for h in range(8):
        np.testing.assert_allclose(got[1, h], v1[h], rtol=0, atol=1e-6)
    assert_close(got, expect, TOL["bf16"], "ctx 0/1/2")


def test_long_split_fp8_matches(pa, cuda):
    case = Case(batch=2, hq=64, hkv=8, d=128, bs=16, kv_dtype="fp8_e4m3", q_dtype="bf16", ctx=[8192, 5001],
                seed=5, partition=512)
    got, expect = _run(pa, cuda, case)
    assert_close(got, expect, TOL["fp8_e4m3"], "fp8 split")


def test_device_flags_for_bad_device_values(pa, cuda):
    case = Case(batch=2, hq=8, hkv=2, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[40, 20], seed=2)
    desc = case.desc(pa)
    kc, vc = case.gpu_pools(pa, cuda)
    status = pa.new_status(cuda)
    # append: one slot negative, one past the pool -> skipped, flagged, other rows written
    k = torch.zeros((3, 2, 128), dtype=torch.bfloat16, device=cuda)
    before = kc.clone()
    slots = torch.tensor([-1, case.num_blocks * 16, 5], dtype=torch.int64, device=cuda)
    pa.kv_append(desc, k, k, slots, kc, vc, status=status)
    assert pa.read_device_status(status) == 1
    changed = (kc.view(torch.int16) != before.view(torch.int16)).any(dim=-1).nonzero().tolist()
    assert all(b == 0 and o == 5 for b, _, o in changed)
    # decode: a block id out of range and a context beyond the table
    bt = torch.from_numpy(case.tables).to(cuda)
    bt[0, 1] = case.num_blocks + 7
    cl = torch.tensor([40, 10_000], dtype=torch.int32, device=cuda)
    q = to_torch(case.q_store, "bf16", cuda)
    for part in (-1, 16):
        out = pa.decode_attention(desc, q, kc, vc, bt, cl, case.scale, partition=part, status=status)
        torch.cuda.synchronize()
        flags = pa.read_device_status(status)
        assert flags & 2 and flags & 4      # the output of such a call is unspecified


def test_copy_blocks(pa, cuda):
    case = Case(batch=1, hq=8, hkv=2, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[64], seed=4,
                spare_blocks=4)
    desc = case.desc(pa)
    kc, vc = case.gpu_pools(pa, cuda)
    src = torch.tensor([int(case.tables[0, 0]), int(case.tables[0, 2])], dtype=torch.int32, device=cuda)
    spare = sorted(set(range(case.num_blocks)) - set(case.tables[0].tolist()))
    dst = torch.tensor(spare[:2], dtype=torch.int32, device=cuda)
    status = pa.new_status(cuda)
    pa.copy_blocks(desc, kc, vc, src, dst, status=status)
    assert pa.read_device_status(status) == 0
    for s, d_ in zip(src.tolist(), dst.tolist()):
        assert torch.equal(kc[d_].view(torch.int16), kc[s].view(torch.int16))
        assert torch.equal(vc[d_].view(torch.int16), vc[s].view(torch.int16))
    bad = torch.tensor([case.num_blocks], dtype=torch.int32, device=cuda)
    pa.copy_blocks(desc, kc, vc, bad, dst[:1], status=status)
    assert pa.read_device_status(status) == 2


def test_fp8_append_is_bit_exact_on_edge_values(pa, cuda):
    # saturation, ties, subnormals, negative zero: the library's quantiser against the oracle's encoder
    vals = np.array([0.0, -0.0, 1e-9, -1e-9, 2.0 ** -10, 3 * 2.0 ** -10, 1.0625, 1.1875, 447.9, 448.0, 464.0,
                     1e6, -1e6, -2.0 ** -10, 0.3, -7.7], dtype=np.float32)
    d = 64
    src = np.resize(vals, (1, 1, d)).astype(np.float32)
    for scale in (1.0, 0.0123):
        case_desc = pa.CacheDesc(2, 16, 1, d, "fp8_e4m3", scale, scale)
        kc, vc = case_desc.new_pools(cuda, fill=0)
        t = torch.from_numpy(src).to(cuda)
        pa.kv_append(case_desc, t, t, torch.tensor([17], dtype=torch.int64, device=cuda), kc, vc)
        got = kc[1, 0, 1].cpu().numpy()
        from oracle import e4m3
        assert np.array_equal(got, e4m3.quantize(src[0, 0], scale))


@pytest.mark.parametrize("partition", [64, 512])   # 47 partitions: merge kernel; 6: fused merge
def test_workspace_counters_return_to_zero_and_reuse(pa, cuda, partition):
    case = Case(batch=3, hq=8, hkv=2, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[3000, 700, 1], seed=9)
    kc, vc = case.gpu_pools(pa, cuda)
    kp, vp = case.oracle_pools()
    expect = case.oracle_out(kp, vp)
    desc = case.desc(pa)
    need = pa.decode_workspace_size(desc, 3, 8, case.max_blocks, partition)
    ws = pa.new_workspace(need, cuda)
    q = to_torch(case.q_store, "bf16", cuda)
    bt = torch.from_numpy(case.tables).to(cuda)
    cl = torch.from_numpy(case.ctx).to(cuda)
    for _ in range(3):   # the same workspace, call after call
        out = pa.decode_attention(desc, q, kc, vc, bt, cl, case.scale, partition=partition, workspace=ws)
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), expect, TOL["bf16"], f"reuse P={partition}")
        counters = ws[:256].view(torch.int32)          # the merge tickets
        assert int(counters.abs().sum()) == 0


def test_large_batch(pa, cuda):
    # 1100 sequences: more than a thread block's worth of per-sequence state anywhere
    rng = np.random.default_rng(13)
    ctx = rng.integers(0, 70, 1100)
    case = Case(batch=1100, hq=8, hkv=2, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=ctx, seed=13)
    got, expect = _run(pa, cuda, case, partition=32)
    assert_close(got, expect, TOL["bf16"], "batch 1100")
