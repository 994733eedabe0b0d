"""The allocation-free decode entry point, for callers that cannot allocate
device memory (a host framework that owns every device allocation, a decode
loop that must not stall on cudaMalloc's device synchronisation, a fixed
footprint).  Its output must match the oracle, and the ordinary entry point,
call after call, while its workspace is the library's own static array that
every call shares.

This file is collected last on purpose: a run that stops at the first
failure has then already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

from harness import TOL, Case, assert_close, to_torch

pytestmark = pytest.mark.gpu


def _inputs(pa, cuda, case):
    kc, vc = case.gpu_pools(pa, cuda)
    q = to_torch(case.q_store, case.q_dtype, cuda)
    bt = torch.from_numpy(case.tables).to(cuda)
    cl = torch.from_numpy(case.ctx).to(cuda)
    return kc, vc, q, bt, cl


def _noalloc_call(pa, case, q, kc, vc, bt, cl, partition, out):
    """One call straight through the C ABI (no binding-side allocation)."""
    from paged_kv_cache_257_gb300 import _native
    c = case.desc(pa).c()
    return _native.lib().pa_decode_attention_noalloc(
        ctypes.byref(c), q.data_ptr(), _native.DTYPE[case.q_dtype], case.hq, kc.data_ptr(), vc.data_ptr(),
        bt.data_ptr(), bt.shape[1], cl.data_ptr(), case.batch, case.scale, partition, out.data_ptr(),
        _native.DTYPE["f32"], None, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _expected(pa, case, kc, vc, qt, bt, cl, partition):
    """(oracle rows, the ordinary entry point's rows) for the case."""
    kp, vp = case.oracle_pools()
    ordinary = pa.decode_attention(case.desc(pa), qt, kc, vc, bt, cl, case.scale, partition=partition)
    return case.oracle_out(kp, vp), ordinary.cpu().numpy()


@pytest.mark.parametrize("kv,q,partition,kernel", [("bf16", "bf16", 256, "auto"),    # few partitions: fused merge
                                                    ("bf16", "bf16", 32, "auto"),     # many partitions: merge kernel
                                                    ("fp8_e4m3", "bf16", 512, "auto"),
                                                    ("fp8_e4m3", "bf16", 512, "warp"),  # one warp per work item
                                                    ("bf16", "bf16", 32, "warp"),
                                                    ("f32", "f32", 64, "auto")])      # CUDA-core kernel
def test_noalloc_matches_the_oracle_and_the_ordinary_entry_point_twice(pa, cuda, kv, q, partition, kernel):
    prev = pa.set_decode_kernel(kernel)
    try:
        _noalloc_against_oracle(pa, cuda, kv, q, partition)
    finally:
        pa.set_decode_kernel(prev)


def _noalloc_against_oracle(pa, cuda, kv, q, partition):
    case = Case(batch=4, hq=16, hkv=4, d=128, bs=16, kv_dtype=kv, q_dtype=q, ctx=[3000, 700, 1, 129], seed=21)
    kc, vc, qt, bt, cl = _inputs(pa, cuda, case)
    oracle, ordinary = _expected(pa, case, kc, vc, qt, bt, cl, partition)
    for call in range(2):   # the static workspace keeps the first call's contents for the second
        out = torch.full((case.batch, case.hq, case.d), float("nan"), dtype=torch.float32, device=cuda)
        st = _noalloc_call(pa, case, qt, kc, vc, bt, cl, partition, out)
        assert st == 0, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert_close(got, oracle, TOL[kv], f"no-alloc call {call} against the oracle")
        assert_close(got, ordinary, TOL[kv], f"no-alloc call {call} against pa_decode_attention")


def test_noalloc_two_shapes_back_to_back_share_the_array(pa, cuda):
    """Two problems of different shapes, split differently (fused merge, then
    the merge kernel, then the first again), one after another on the shared
    array: each call clears the counters it needs and lays out its own
    partials, whatever the previous call left there."""
    a = Case(batch=3, hq=32, hkv=8, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[4000, 17, 2500], seed=5)
    b = Case(batch=5, hq=8, hkv=1, d=128, bs=32, kv_dtype="f16", q_dtype="f16", ctx=[64, 1, 900, 2048, 333],
             seed=6)
    runs = []
    for case, partition in ((a, 512), (b, 64)):
        kc, vc, qt, bt, cl = _inputs(pa, cuda, case)
        oracle, _ = _expected(pa, case, kc, vc, qt, bt, cl, partition)
        runs.append((case, partition, (kc, vc, qt, bt, cl), oracle))
    for case, partition, (kc, vc, qt, bt, cl), oracle in runs + runs[:1]:
        out = torch.full((case.batch, case.hq, case.d), float("nan"), dtype=torch.float32, device=cuda)
        assert _noalloc_call(pa, case, qt, kc, vc, bt, cl, partition, out) == 0
        torch.cuda.synchronize()
        assert_close(out.cpu().numpy(), oracle, TOL[case.kv_dtype], f"{case.kv_dtype} batch {case.batch}")


def test_noalloc_rejects_workspaces_beyond_its_array(pa, cuda):
    # 4 x 64 heads x 256 partitions of 512 tokens need ~34 MB of partials: more than the 8 MiB array
    from paged_kv_cache_257_gb300 import _native
    desc = pa.CacheDesc(32768, 16, 8, 128, "fp8_e4m3", 0.01, 0.01)
    assert pa.decode_workspace_size(desc, 4, 64, 8192, 512) > _native.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((4, 64, 128), dtype=torch.bfloat16, device=cuda)
    bt = torch.zeros((4, 8192), dtype=torch.int32, device=cuda)
    cl = torch.zeros(4, dtype=torch.int32, device=cuda)
    out = torch.zeros((4, 64, 128), dtype=torch.float32, device=cuda)
    with pytest.raises(pa.NativeError) as e:
        pa.decode_attention_noalloc(desc, q, q, q, bt, cl, 0.088, out, partition=512)
    assert e.value.status == "PA_ERR_RANGE"
    assert np.all(out.cpu().numpy() == 0)          # nothing was launched
    with pytest.raises(ValueError):
        pa.decode_attention_noalloc(desc, q, q, q, bt, cl, 0.088, None, partition=512)
