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
