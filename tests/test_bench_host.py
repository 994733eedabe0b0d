"""Host-side pieces of bench.py that need no GPU: the fingerprint that keys
recorded ncu traffic to the kernel code, and the recorded traffic itself."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _fingerprint_of(tmp_path, text):
    f = tmp_path / "k.cu"
    f.write_text(text)
    return bench._code_fingerprint([str(f)])


def test_fingerprint_ignores_comments_and_white_space(tmp_path):
    base = _fingerprint_of(tmp_path, "int f(int x) {\n    return x + 1;\n}\n")
    assert _fingerprint_of(tmp_path, "// a note\nint f(int x) {   return x + 1; /* why */ }\n") == base
    assert _fingerprint_of(tmp_path, "int f(int x)\n{\n\treturn x + 1;  // one more\n}\n") == base


def test_fingerprint_follows_the_code(tmp_path):
    base = _fingerprint_of(tmp_path, "int f(int x) { return x + 1; }\n")
    assert _fingerprint_of(tmp_path, "int f(int x) { return x + 2; }\n") != base
    # conservative: joining tokens counts as an edit (counters may be voided
    # by a format-only change, never kept across a code change)
    assert _fingerprint_of(tmp_path, "int f(int x) { return x+1; }\n") != base


def test_recorded_traffic_is_consistent():
    """Counters recorded for the current kernel code (none after a code
    change, until a new capture) cover at least each workload's algorithmic
    KV bytes and at most 2% more: no re-reads."""
    import pytest
    algorithmic = {"gqa_bf16": 281_624_576, "mha_f16": 671_088_640, "longctx_fp8": 1_073_741_824}
    recorded = {w: bench.captured_traffic(w) for w in algorithmic}
    if all(t is None for t in recorded.values()):
        pytest.skip("no ncu capture recorded for the current kernel code")
    for w, kv in algorithmic.items():
        assert recorded[w] is not None and kv <= recorded[w] <= kv * 1.02, (w, recorded[w])
        # the KV loads move whole 128-byte lines: four 32-byte sectors per L2 request
        spr = bench.captured_sectors_per_request(w)
        assert spr is not None and 3.9 <= spr <= 4.0, (w, spr)


def test_oracle_sample_reads_the_workloads_own_tokens():
    """The oracle baseline's compact sample (a share of the sequences, block
    ids renumbered) attends to exactly the tokens the full workload holds:
    its rows equal the oracle's rows over the whole tiny workload."""
    import numpy as np
    from oracle import attention as oatt
    from oracle import cache as ocache
    from synth import workloads as wl
    w = wl.make("tiny")
    kp = ocache.new_pool(w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim, w.kv_dtype)
    vp = ocache.new_pool(w.num_blocks, w.n_kv_heads, w.block_size, w.head_dim, w.kv_dtype)
    for s, n in enumerate(w.context_lens):
        slots = ocache.slot_mapping(w.block_tables, [s] * int(n), range(int(n)), w.block_size)
        ocache.kv_append(kp, vp, wl.kv_tokens_f32(w, "k", s, 0, int(n)), wl.kv_tokens_f32(w, "v", s, 0, int(n)),
                         slots, "f32", "f32")
    full = oatt.decode_attention_paged(wl.queries_f32(w), kp, vp, w.block_tables, w.context_lens, w.scale, "f32")
    seqs, cap = bench.oracle_share("tiny", 1, 2)
    assert seqs == [1, 3] and cap is None
    s = bench.oracle_sample("tiny", seqs, cap)
    assert s["units"] == 2.0 and s["kp"].shape[0] == sum(-(-int(w.context_lens[i]) // 16) for i in seqs)
    part = oatt.decode_attention_paged(s["q"], s["kp"], s["vp"], s["tables"], s["ctx"], w.scale, "f32")
    assert np.array_equal(part, full[seqs])


def test_oracle_share_caps_long_contexts():
    seqs, cap = bench.oracle_share("longctx_fp8", 5, 16)
    assert seqs == [1] and cap == bench.ORACLE_TOKEN_CAP
    assert bench.oracle_share("gqa_bf16", 3, 16) == ([3, 19], None)
