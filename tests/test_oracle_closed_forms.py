"""Pins for oracle.closed_forms: values printed on the pages, and invariants."""

import os

import numpy as np
import pytest

from oracle import closed_forms as cf

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_bytes_per_token_worked_examples():
    rows = _rows("bytes_per_token.txt")
    per_token = {r[0]: r for r in rows if len(r) == 6}
    assert set(per_token) == {"llama2_13b_fp16", "llama3_8b_fp16"}
    for name, layers, hkv, d, b, expect in per_token.values():
        assert cf.kv_bytes_per_token(int(layers), int(hkv), int(d), int(b)) == int(expect), name


def test_request_and_batch_sizes_from_example_2():
    rows = {r[0]: r for r in _rows("bytes_per_token.txt") if len(r) == 4}
    per_tok = cf.kv_bytes_per_token(32, 8, 128, 2)
    for name, tokens, batch, expect in rows.values():
        assert int(tokens) * int(batch) * per_tok == int(expect), name
    # Example 1 at 4096 tokens: "approx 800 KB per token" and "approx 3.2 GB per
    # sequence" are rounded figures; the exact product is 3.125 GiB, and 8
    # sequences (the page's 25.6 GB) are exactly 25 GiB
    per13 = cf.kv_bytes_per_token(40, 40, 128, 2)
    assert per13 / 1024 == 800.0
    assert 4096 * per13 == 3_355_443_200 == int(3.125 * 2**30)
    assert 8 * 4096 * per13 == 25 * 2**30


def test_fp8_halves_the_cache():
    # FP8 KV stores one byte where FP16 stores two: half the bytes per token
    for layers, hkv, d in ((40, 40, 128), (32, 8, 128), (80, 8, 128)):
        assert 2 * cf.kv_bytes_per_token(layers, hkv, d, 1) == cf.kv_bytes_per_token(layers, hkv, d, 2)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_tail_waste_confined_to_last_block(bs):
    for n in range(0, 5 * bs + 1):
        blocks = cf.blocks_for_tokens(n, bs)
        waste = cf.tail_waste_slots(n, bs)
        assert 0 <= waste <= bs - 1
        assert blocks * bs >= n
        assert n == 0 or (blocks - 1) * bs < n


def test_mean_tail_is_about_eight_tokens_at_block_16():
    # "the average unused tail is ~8 tokens" over sequences of varying lengths
    lengths = np.arange(1, 100_001)
    mean_tail = np.mean([cf.tail_waste_slots(int(n), 16) for n in lengths[::7]])
    assert 7.0 < mean_tail < 8.0


def test_kv_bytes_for_sequences_tiny_and_mha():
    # tiny workload: contexts {5,17,33,64}, Hkv=2, D=64, float32
    assert cf.kv_bytes_for_sequences([5, 17, 33, 64], 2, 64, 4) == 121_856
    # Llama-2-13B-shaped layer, 8 x 4096 tokens, fp16
    assert cf.kv_bytes_for_sequences([4096] * 8, 40, 128, 2) == 671_088_640
    # 70B-shaped long context, 4 x 131072 tokens, FP8
    assert cf.kv_bytes_for_sequences([131072] * 4, 8, 128, 1) == 1_073_741_824


def test_rejects_bad_sizes():
    with pytest.raises(ValueError):
        cf.blocks_for_tokens(5, 0)
    with pytest.raises(ValueError):
        cf.kv_bytes_per_token(1.5, 8, 128, 2)
