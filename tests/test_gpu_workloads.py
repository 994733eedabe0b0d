"""Parity at full size: the bench's own workloads, built and launched exactly
as bench.py times them (its set-up, its partition choice, one step of append
plus decode), checked on sampled sequences against the oracle.

The expected values come from the workloads' synthetic token values, stored
by the oracle's own quantisation and passed through the plain attention
definition in float64 ([DEV] section 1 and section 2 Example 2); nothing is
read back from the device but the outputs under test."""

import os
import sys

import numpy as np
import pytest

from harness import TOL, assert_close
from oracle import attention as oatt
from oracle import numerics
from synth import workloads as wl

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _sample(ctx, k):
    """Indices of the longest (k = 1), or of the shortest, the longest and
    evenly spread others."""
    order = np.argsort(ctx, kind="stable")
    if k == 1:
        return [int(order[-1])]
    picks = {int(order[0]), int(order[-1])}
    for i in np.linspace(0, len(ctx) - 1, k):
        picks.add(int(order[int(i)]))
    return sorted(picks)[:k]


def _oracle_row(w, wk, s):
    n = int(wk.ctx_decode[s])
    q = numerics.to_f64(wl.cast(wl.queries_f32(w), w.q_dtype)[s], w.q_dtype)
    kv = []
    for which, scale in (("k", wk.desc.k_scale), ("v", wk.desc.v_scale)):
        src = wl.cast(wl.kv_tokens_f32(w, which, s, 0, n), w.src_dtype)
        stored = numerics.store(src, w.src_dtype, w.kv_dtype, scale)
        kv.append(numerics.to_f64(stored, w.kv_dtype, scale))
    return oatt.decode_attention_contiguous(q, kv[0], kv[1], w.scale)


@pytest.mark.parametrize("name,k", [("gqa_bf16", 4), ("mha_f16", 2), ("prefix_bf16", 3), ("longctx_fp8", 1)])
def test_bench_workload_step_matches_oracle(pa, cuda, name, k):
    sys.path.insert(0, ROOT)
    import bench
    wk = bench.GpuWorkload(name, cuda, replicas=1)
    w = wk.w
    wk.step(0)
    import torch
    torch.cuda.synchronize()
    out = wk.out.cpu().numpy()
    for s in _sample(wk.ctx_decode, k):
        assert_close(out[s], _oracle_row(w, wk, s), TOL[w.kv_dtype], f"{name} sequence {s}")
