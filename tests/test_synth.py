"""The seeded input generator: determinism, counter-based sub-ranges, distribution
and the workloads' shapes."""

import numpy as np

import synth
from synth import workloads


def test_counter_based_subranges_agree():
    full = synth.normal_f32(3, 77, 10_000)
    part = synth.normal_f32(3, 77, 1000, offset=4000)
    assert np.array_equal(full[4000:5000], part)
    assert np.array_equal(full, synth.normal_f32(3, 77, 10_000))
    assert not np.array_equal(full, synth.normal_f32(3, 78, 10_000))


def test_normal_moments():
    x = synth.normal_f64(1, 1, 2_000_000)
    assert abs(x.mean()) < 3e-3 and abs(x.std() - 1) < 3e-3
    assert abs(np.mean(x ** 4) - 3) < 0.05


def test_integer_draws_match_the_published_finaliser():
    # h(k, i) = mix64(k + (i+1) * golden) with k = mix64(seed + (stream+1) * golden)
    def mix(z):
        m = (1 << 64) - 1
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
        return z ^ (z >> 31)
    g, m = 0x9E3779B97F4A7C15, (1 << 64) - 1
    k = mix((5 + 2 * g) & m)
    expect = [mix((k + (i + 1) * g) & m) for i in range(4)]
    assert list(synth.u64(5, 1, 4)) == expect


def test_workload_shapes():
    t = workloads.make("tiny")
    assert list(t.context_lens) == [5, 17, 33, 64] and t.num_blocks == 32
    used = t.block_tables[t.block_tables >= 0]
    assert len(set(t.block_tables[0, :1]) | set(t.block_tables[1, :2]) | set(t.block_tables[2, :3])
               | set(t.block_tables[3, :4])) == 10
    g = workloads.make("gqa_bf16")
    assert g.batch == 32 and g.context_lens.min() >= 1 and g.context_lens.max() <= 4096
    blocks = sum(-(-int(c) // 16) for c in g.context_lens)
    assert g.num_blocks == blocks + 32
    flat = np.concatenate([g.block_tables[s, :-(-int(c) // 16)] for s, c in enumerate(g.context_lens)])
    assert len(np.unique(flat)) == blocks                 # a partition: no block used twice
    slots = workloads.append_slots(g)
    assert len(np.unique(slots)) == 32
    f = workloads.make("longctx_fp8")
    assert f.num_blocks == 32768 and f.partition_size == 512 and f.q_dtype == "bf16"
    p = workloads.make("prefix_bf16")
    assert p.block_tables is None and p.prefix_len == 2048 and p.context_lens.min() > 2048


def test_prefix_tokens_are_shared_between_sequences():
    p = workloads.make("prefix_bf16")
    a = workloads.kv_tokens_f32(p, "k", 0, 2040, 2050)
    b = workloads.kv_tokens_f32(p, "k", 1, 2040, 2050)
    assert np.array_equal(a[:8], b[:8]) and not np.array_equal(a[8:], b[8:])
