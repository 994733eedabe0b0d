"""Parity at full size: the bench's own workloads, built and launched exactly
as bench.py times them (its set-up, its partition choice, one step of append
plus decode), every sequence of the batch checked against the oracle, under
both decode schedules (the default balanced tail and the bit-reproducible
fixed one).

The expected values come from the workloads' synthetic token values, stored
by the oracle's own quantisation and passed through the plain attention
definition in float64 ([DEV] section 1 and section 2 Example 2); nothing is
read back from the device but the outputs under test."""

import multiprocessing as mp
import os
import sys

import numpy as np
import pytest

from harness import TOL, assert_close

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _oracle_row(name, s, n, k_scale, v_scale):
    """Expected output rows of sequence ``s`` over its ``n`` cached tokens."""
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    from oracle import attention as oatt
    from oracle import numerics
    from synth import workloads as wl
    w = wl.make(name)
    q = numerics.to_f64(wl.cast(wl.queries_f32(w), w.q_dtype)[s], w.q_dtype)
    kv = []
    for which, scale in (("k", k_scale), ("v", v_scale)):
        src = wl.cast(wl.kv_tokens_f32(w, which, s, 0, n), w.src_dtype)
        stored = numerics.store(src, w.src_dtype, w.kv_dtype, scale)
        kv.append(numerics.to_f64(stored, w.kv_dtype, scale))
    return oatt.decode_attention_contiguous(q, kv[0], kv[1], w.scale)


def _oracle_rows(name, wk):
    """Every sequence's expected rows; the 128k-token sequences of the long
    context workload are computed in spawned processes, one per sequence."""
    args = [(name, s, int(wk.ctx_decode[s]), wk.desc.k_scale, wk.desc.v_scale) for s in range(wk.w.batch)]
    if max(a[2] for a in args) <= 8192:
        return [_oracle_row(*a) for a in args]
    n = len(args)
    threads = str(max(1, (os.cpu_count() or 1) // n))
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS")}
    os.environ.update(OPENBLAS_NUM_THREADS=threads, OMP_NUM_THREADS=threads)
    try:
        with mp.get_context("spawn").Pool(n) as pool:
            return pool.starmap(_oracle_row, args)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("name", ["gqa_bf16", "mha_f16", "prefix_bf16", "longctx_fp8", "tiny"])
def test_bench_workload_step_matches_oracle(pa, cuda, name):
    sys.path.insert(0, ROOT)
    import bench
    import torch
    wk = bench.GpuWorkload(name, cuda, replicas=1)
    expect = _oracle_rows(name, wk)
    prev = pa.decode_deterministic()
    try:
        for deterministic in (False, True):
            pa.set_decode_deterministic(deterministic)
            wk.out.fill_(float("nan"))
            wk.step(0)
            torch.cuda.synchronize()
            out = wk.out.cpu().numpy()
            for s in range(wk.w.batch):
                assert_close(out[s], expect[s], TOL[wk.w.kv_dtype],
                             f"{name} sequence {s} ({'fixed' if deterministic else 'balanced'} schedule)")
    finally:
        pa.set_decode_deterministic(prev)
