"""Seeded random configurations through the whole decode path against the
oracle: dtypes, GQA groupings (including more than 8 query heads per KV
head), head sizes, block sizes, partition sizes, ragged and empty contexts
and slid windows, drawn from one seed per case so that a failure names a
reproducible configuration."""

import numpy as np
import pytest
import torch

from harness import TOL, Case, assert_close, to_torch
from oracle import attention as oatt

pytestmark = pytest.mark.gpu

PAIRS = [("bf16", "bf16"), ("f16", "f16"), ("fp8_e4m3", "bf16"), ("fp8_e4m3", "f16"), ("f32", "f32"),
         ("bf16", "f32"), ("f16", "bf16")]


def _config(seed):
    rng = np.random.default_rng(1000 + seed)
    kv, q = PAIRS[rng.integers(len(PAIRS))]
    hkv = int(rng.choice([1, 2, 4, 8]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    d = 128 if rng.random() < 0.8 else int(rng.choice([64, 256]))
    bs = int(rng.choice([8, 16, 32]))
    batch = int(rng.integers(1, 9))
    cap = int(rng.choice([64, 700, 3000]))
    ctx = [int(x) for x in rng.integers(0, cap + 1, batch)]
    ctx[rng.integers(batch)] = cap                       # at least one sequence fills its table
    partition = int(rng.choice([0, -1, 16, 64, 256, 1024]))
    if partition > 0:                                    # a multiple of the partition unit
        partition = -(-partition // max(16, bs)) * max(16, bs)
    window = rng.random() < 0.3
    starts = [int(rng.integers(0, c + 1)) for c in ctx] if window else None
    return dict(kv=kv, q=q, hkv=hkv, hq=hkv * g, d=d, bs=bs, batch=batch, ctx=ctx, partition=partition,
                starts=starts)


@pytest.mark.parametrize("kernel", ["cta", "warp"], indirect=True)
@pytest.mark.parametrize("seed", range(100))
def test_random_configuration(pa, cuda, kernel, seed):
    c = _config(seed)
    case = Case(batch=c["batch"], hq=c["hq"], hkv=c["hkv"], d=c["d"], bs=c["bs"], kv_dtype=c["kv"], q_dtype=c["q"],
                ctx=c["ctx"], seed=2000 + seed)
    kc, vc = case.gpu_pools(pa, cuda)
    status = pa.new_status(cuda)
    starts = None if c["starts"] is None else torch.tensor(c["starts"], dtype=torch.int32, device=cuda)
    out = pa.decode_attention(case.desc(pa), to_torch(case.q_store, case.q_dtype, cuda), kc, vc,
                              torch.from_numpy(case.tables).to(cuda), torch.from_numpy(case.ctx).to(cuda),
                              case.scale, partition=c["partition"], status=status, context_starts=starts)
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0, c
    kp, vp = case.oracle_pools()
    want = oatt.decode_attention_paged(case.q_store, kp, vp, case.tables, case.ctx, case.scale, case.kv_dtype,
                                       case.k_scale, case.v_scale, q_dtype=case.q_dtype, context_starts=c["starts"])
    assert_close(out.cpu().numpy(), want, TOL[c["kv"]], f"{c} {kernel}")
