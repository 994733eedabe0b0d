"""GPU parity of decode over block tables built by the prefix cache.

[DEV] section 5, 2 "Automatic Prefix Caching": a request whose prompt
matches a computed sequence maps the cached physical blocks into its table
and skips their prefill.  Each token's K/V here is drawn from a seed that
depends on the whole token prefix up to it (as a model's would), so a mapped
block must hold exactly what the request would have computed.  Decode over
the cache-built tables is compared with attention over each request's K/V
generated directly, with no cache."""

import numpy as np
import pytest
import torch

import synth
from harness import POISON, TOL, assert_close, to_torch
from oracle import attention as oatt
from oracle import numerics
from oracle.prefix_cache import fnv1a64
from synth import workloads

pytestmark = pytest.mark.gpu

BS, HKV, HQ, D = 16, 2, 8, 128


def _kv_of(tokens):
    """[n, HKV, D] bf16 K and V whose row p depends on tokens[: p + 1]."""
    ks, vs, h = [], [], 0xcbf29ce484222325
    for t in tokens:
        h = fnv1a64(int(t).to_bytes(4, "little"), h)
        ks.append(synth.normal_f32(80, (h >> 1) & ((1 << 62) - 1), HKV * D))
        vs.append(synth.normal_f32(81, (h >> 1) & ((1 << 62) - 1), HKV * D))
    shape = (len(tokens), HKV, D)
    return workloads.cast(np.stack(ks).reshape(shape), "bf16"), workloads.cast(np.stack(vs).reshape(shape), "bf16")


def test_decode_over_prefix_cached_tables(pa, cuda):
    rng = np.random.default_rng(12)
    nb = 128
    alloc = pa.BlockAllocator(nb, 6)
    cache = pa.PrefixCache(alloc, BS)
    desc = pa.CacheDesc(nb, BS, HKV, D, "bf16", 1.0, 1.0)
    kc, vc = desc.new_pools(cuda, fill=POISON)
    prompts = [list(map(int, rng.integers(0, 1000, 64))), list(map(int, rng.integers(0, 1000, 40)))]
    requests, rows, lens, matched = [], [], [], 0
    for r in range(10):
        toks = prompts[r % 2] + list(map(int, rng.integers(0, 1000, int(rng.integers(1, 40)))))
        row = [-1] * 8
        m = cache.match(toks, row)
        matched += m
        n = m
        slots = []
        for t in range(m * BS, len(toks)):          # prefill only what the cache did not hold
            slot, n, _ = alloc.append_slot(row, n, t, BS)
            slots.append(slot)
        k, v = _kv_of(toks)
        pa.kv_append(desc, to_torch(k[m * BS:], "bf16", cuda), to_torch(v[m * BS:], "bf16", cuda),
                     torch.tensor(slots, dtype=torch.int64, device=cuda), kc, vc)
        cache.insert(toks, row, n)
        requests.append((toks, k, v)), rows.append(row), lens.append(len(toks))
    assert matched >= 8 * 2          # every request after the first of its prompt maps the prompt's full blocks
    q_store = workloads.cast(synth.normal_f32(82, 1, 10 * HQ * D).reshape(10, HQ, D), "bf16")
    status = pa.new_status(cuda)
    out = pa.decode_attention(desc, to_torch(q_store, "bf16", cuda), kc, vc,
                              torch.tensor(np.array(rows, np.int32), device=cuda),
                              torch.tensor(lens, dtype=torch.int32, device=cuda), 1 / np.sqrt(D), status=status)
    torch.cuda.synchronize()
    assert pa.read_device_status(status) == 0
    qf = numerics.to_f64(q_store, "bf16")
    for i, (toks, k, v) in enumerate(requests):
        want = oatt.decode_attention_contiguous(qf[i], numerics.to_f64(k, "bf16"), numerics.to_f64(v, "bf16"),
                                                1 / np.sqrt(D))
        assert_close(out[i].cpu().numpy(), want, TOL["bf16"], f"request {i}")
    # memory: the prompts' full blocks are held once, not per request
    used = nb - alloc.free_count
    private = sum(-(-ln // BS) for ln in lens)
    assert used < private
