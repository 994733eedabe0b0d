"""Parity at the library's size limits, against the oracle: the largest
partition count a call may have (32768, merged by the merge kernel) and the
largest batch (65535 sequences, the grid's z extent), under both
tensor-core kernels."""

import numpy as np
import pytest

from harness import TOL, Case, assert_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_maximum_partition_count(pa, cuda, kernel):
    """One sequence of 524288 tokens in 16-token partitions: 32768 partials."""
    ctx = 32768 * 16
    case = Case(batch=1, hq=8, hkv=1, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=[ctx], seed=61,
                spare_blocks=1)
    assert -(-case.max_blocks * case.bs // 16) == 32768
    kc, vc = case.gpu_pools(pa, cuda)
    status = pa.new_status(cuda)
    out = case.gpu_decode(pa, cuda, kc, vc, partition=16, status=status)
    assert pa.read_device_status(status) == 0
    kp, vp = case.oracle_pools()
    assert_close(out.cpu().numpy(), case.oracle_out(kp, vp), TOL["bf16"], f"32768 partitions {kernel}")


@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
def test_maximum_batch(pa, cuda, kernel):
    """65535 sequences of 0 to 40 tokens (one or two 32-token partitions)."""
    rng = np.random.default_rng(62)
    ctx = rng.integers(0, 41, 65535)
    case = Case(batch=65535, hq=2, hkv=1, d=128, bs=16, kv_dtype="bf16", q_dtype="bf16", ctx=ctx, seed=62)
    kc, vc = case.gpu_pools(pa, cuda)
    status = pa.new_status(cuda)
    out = case.gpu_decode(pa, cuda, kc, vc, partition=32, status=status)
    assert pa.read_device_status(status) == 0
    got = out.cpu().numpy()
    assert np.array_equal(got[ctx == 0], np.zeros_like(got[ctx == 0]))
    kp, vp = case.oracle_pools()
    assert_close(got, case.oracle_out(kp, vp), TOL["bf16"], f"batch 65535 {kernel}")
