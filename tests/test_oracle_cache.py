"""Pins for oracle.cache and oracle.numerics: the block-table diagram printed on
the pages, append/gather round trips, and torch's bf16 rounding."""

import os

import numpy as np
import pytest
import torch

from oracle import cache, e4m3, numerics

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _diagram():
    with open(os.path.join(GOLDEN, "block_table_diagram.txt")) as f:
        return [tuple(int(v) for v in ln.split()) for ln in f if ln.strip() and not ln.startswith("#")]


def test_slot_mapping_follows_the_block_table_diagram():
    rows = _diagram()
    table = [phys for _, _, _, phys in rows]
    assert table == [84, 12, 903]
    for logical, first, last, phys in rows:
        for p in range(first, last + 1):
            assert p // 16 == logical
            assert cache.slot_of(table, p, 16) == phys * 16 + (p - first)
    slots = cache.slot_mapping([table], [0] * 48, list(range(48)), 16)
    assert slots.dtype == np.int64
    assert list(slots[:3]) == [84 * 16, 84 * 16 + 1, 84 * 16 + 2]
    assert slots[16] == 12 * 16 and slots[47] == 903 * 16 + 15


def test_slot_mapping_rejects_positions_beyond_table():
    with pytest.raises(ValueError):
        cache.slot_of([3, 4], 32, 16)
    with pytest.raises(ValueError):
        cache.slot_of([3, 4], -1, 16)


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_append_then_gather_round_trips(dtype):
    rng = np.random.default_rng(1)
    nb, hkv, bs, d = 12, 3, 16, 8
    table = [7, 2, 11]
    ctx = 37
    vals = rng.normal(size=(ctx, hkv, d)).astype(np.float32)
    src = numerics.store(vals, "f32", dtype)         # values representable in the cache type
    kp = cache.new_pool(nb, hkv, bs, d, dtype)
    vp = cache.new_pool(nb, hkv, bs, d, dtype)
    before = kp.copy()
    slots = cache.slot_mapping([table], [0] * ctx, range(ctx), bs)
    cache.kv_append(kp, vp, src, src, slots, dtype, dtype)
    got = cache.gather_logical(kp, table, ctx)
    assert np.array_equal(got.view(np.uint8), np.asarray(src).view(np.uint8))
    # untouched blocks and tail slots keep their contents
    untouched = np.ones(nb * bs, dtype=bool)
    untouched[slots] = False
    flat_after = kp.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d)
    flat_before = before.transpose(0, 2, 1, 3).reshape(nb * bs, hkv, d)
    assert np.array_equal(flat_after[untouched].view(np.uint8), flat_before[untouched].view(np.uint8))


def test_append_fp8_stores_quantised_codes():
    rng = np.random.default_rng(2)
    vals = rng.normal(size=(5, 2, 16)).astype(np.float32)
    s = np.float32(0.01)
    kp = cache.new_pool(4, 2, 16, 16, "fp8_e4m3")
    vp = cache.new_pool(4, 2, 16, 16, "fp8_e4m3")
    slots = np.array([3, 17, 18, 40, 63])
    cache.kv_append(kp, vp, vals, vals, slots, "f32", "fp8_e4m3", s, s)
    ref = torch.from_numpy(vals / s).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t, slot in enumerate(slots):
        b, o = divmod(int(slot), 16)
        assert np.array_equal(kp[b, :, o, :], ref[t])


def test_append_rejects_out_of_range_slots():
    kp = cache.new_pool(2, 1, 16, 4, "f32")
    vp = cache.new_pool(2, 1, 16, 4, "f32")
    x = np.zeros((1, 1, 4), dtype=np.float32)
    for bad in (-1, 32):
        with pytest.raises(ValueError):
            cache.kv_append(kp, vp, x, x, [bad], "f32", "f32")


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.normal(0, 1, 100000), rng.normal(0, 1e30, 1000),
                        rng.normal(0, 1e-30, 1000)]).astype(np.float32)
    # exact ties: low 16 bits == 0x8000, both parities of the kept lsb
    ties = (rng.integers(0, 2**15, 1000, dtype=np.uint32) << 17 | np.uint32(0x8000)).view(np.float32)
    ties2 = (rng.integers(0, 2**15, 1000, dtype=np.uint32) << 17 | np.uint32(0x18000)).view(np.float32)
    x = np.concatenate([x, ties, ties2])
    nan = np.isnan(x)
    assert np.all(np.isnan(numerics.bf16_bits_to_f64(numerics.f32_to_bf16_bits(x[nan]))))
    x = x[~nan]                      # NaN payloads are not part of the path
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(numerics.f32_to_bf16_bits(x), ref)
    back = numerics.bf16_bits_to_f64(ref)
    assert np.array_equal(back, torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


def test_to_f64_fp8_uses_scale():
    codes = np.array([0x38, 0x7E, 0x81], dtype=np.uint8)
    assert list(numerics.to_f64(codes, "fp8_e4m3", np.float32(0.5))) == [0.5, 224.0, -2.0 ** -10]
    assert e4m3.decode(0x81) == -(2.0 ** -9)
