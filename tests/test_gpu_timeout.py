"""A copy that never completes its stage ends in a status, not a hang.

A test build of the library arms every stage for 16 bytes more than its
copies bring (PA_TEST_EXTRA_TX; the copies themselves complete normally), so
each bounded mbarrier wait runs into its one-second limit.  The call must
return, raise PA_DEVFLAG_TIMEOUT in the device status word, and leave the
context usable: the ordinary library then decodes the same inputs correctly."""

import ctypes
import time

import pytest
import torch

from harness import TOL, Case, assert_close, to_torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", ["cta", "warp"])
def test_stalled_stage_times_out_and_the_context_survives(pa, cuda, which):
    from paged_kv_cache_257_gb300 import _native, build
    path = build.build_variant("test_stall", ["-DPA_TEST_EXTRA_TX=16"], ["decode_mma.cu", "decode_warp.cu"])
    stall = _native.load(path)
    assert stall.pa_set_decode_kernel(_native.DECODE_KERNEL[which]) == 0
    # one sequence of one partition: a single CTA, so the waits run out once
    case = Case(batch=1, hq=8, hkv=1, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[100], seed=71)
    kc, vc = case.gpu_pools(pa, cuda)
    q = to_torch(case.q_store, case.q_dtype, cuda)
    bt = torch.from_numpy(case.tables).to(cuda)
    cl = torch.from_numpy(case.ctx).to(cuda)
    out = torch.zeros((1, 8, 128), dtype=torch.float32, device=cuda)
    status = pa.new_status(cuda)
    c = case.desc(pa).c()
    t0 = time.perf_counter()
    st = stall.pa_decode_attention(ctypes.byref(c), q.data_ptr(), _native.DTYPE["bf16"], 8, kc.data_ptr(),
                                   vc.data_ptr(), bt.data_ptr(), bt.shape[1], cl.data_ptr(), 1, case.scale, -1,
                                   None, 0, out.data_ptr(), _native.DTYPE["f32"], status.data_ptr(),
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 30
    assert pa.read_device_status(status) & 8           # PA_DEVFLAG_TIMEOUT
    # the context still works: the ordinary library on the same inputs
    got = pa.decode_attention(case.desc(pa), q, kc, vc, bt, cl, case.scale, partition=-1, status=status)
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0
    kp, vp = case.oracle_pools()
    assert_close(got.cpu().numpy(), case.oracle_out(kp, vp), TOL["bf16"], "after the timeout")
