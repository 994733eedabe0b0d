"""Pins for oracle.e4m3: the OCP E4M3 bit layout, a library decoder/encoder
(torch.float8_e4m3fn), and brute-force nearest-value search."""

import numpy as np
import pytest
import torch

from oracle import e4m3

ALL = np.arange(256, dtype=np.uint8)


def _finite_codes():
    v = e4m3.decode(ALL)
    return ALL[~np.isnan(v)], v[~np.isnan(v)]


def test_decode_anchor_values():
    d = e4m3.decode
    assert d(0x00) == 0.0 and np.signbit(d(0x80))
    assert d(0x01) == 2.0 ** -9            # smallest subnormal
    assert d(0x07) == 7 * 2.0 ** -9        # largest subnormal
    assert d(0x08) == 2.0 ** -6            # smallest normal
    assert d(0x38) == 1.0                  # E=7, M=0
    assert d(0x77) == 240.0                # E=14, M=7
    assert d(0x78) == 256.0                # E=15, M=0 is finite in this variant
    assert d(0x7E) == 448.0                # largest finite
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0xFE) == -448.0


def test_decode_structure():
    codes, vals = _finite_codes()
    assert len(codes) == 254
    pos = e4m3.decode(np.arange(0, 0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)                       # monotone on positive codes
    assert np.array_equal(e4m3.decode(ALL[0x80:0xFF]), -e4m3.decode(ALL[0:0x7F]))


def test_decode_matches_torch_float8():
    t = torch.from_numpy(ALL.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = e4m3.decode(ALL)
    nan = np.isnan(t)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(t[~nan], ours[~nan])


def _brute_force(x):
    """Nearest finite code, ties to the even code, saturating beyond 448."""
    codes, vals = _finite_codes()
    out = []
    for xi in np.atleast_1d(x):
        if xi >= 448.0:
            out.append(0x7E)
            continue
        if xi <= -448.0:
            out.append(0xFE)
            continue
        err = np.abs(vals - xi)
        best = np.flatnonzero(err == err.min())
        cands = [int(codes[i]) for i in best]
        # of the nearest, prefer the sign of x (matters only for zero), then an even code
        same_sign = [c for c in cands if (c >> 7) == int(np.signbit(xi))] or cands
        even = [c for c in same_sign if c % 2 == 0] or same_sign
        out.append(even[0])
    return np.array(out, dtype=np.uint8)


def test_encode_brute_force_dense():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.normal(0, 1, 4000), rng.normal(0, 100, 2000), rng.uniform(-2e-2, 2e-2, 2000),
        rng.uniform(-500, 500, 1000),
    ])
    assert np.array_equal(e4m3.encode(x), _brute_force(x))


def test_encode_exact_midpoints_round_to_even():
    _, vals = _finite_codes()
    pos = np.unique(vals[vals >= 0])
    mids = (pos[:-1] + pos[1:]) / 2
    x = np.concatenate([mids, -mids, pos, -pos])
    assert np.array_equal(e4m3.encode(x), _brute_force(x))
    assert e4m3.encode(2.0 ** -10) == 0x00          # tie between 0 and 2^-9 -> even (0)
    assert e4m3.encode(3 * 2.0 ** -10) == 0x02      # tie between 1 and 2 (x 2^-9) -> 2
    assert e4m3.encode(1.0625) == 0x38              # tie between 1.0 and 1.125 -> 1.0
    assert e4m3.encode(1.1875) == 0x3A              # tie between 1.125 and 1.25 -> 1.25


def test_encode_saturates_and_handles_nan():
    assert list(e4m3.encode([448.0, 449.0, 464.0, 1e6, np.inf])) == [0x7E] * 5
    assert list(e4m3.encode([-449.0, -1e30, -np.inf])) == [0xFE] * 3
    assert e4m3.encode(np.nan) == 0x7F
    assert e4m3.encode(-0.0) == 0x80 and e4m3.encode(-1e-9) == 0x80


def test_encode_matches_torch_within_range():
    rng = np.random.default_rng(11)
    x = np.concatenate([rng.normal(0, 3, 20000), rng.uniform(-447.9, 447.9, 5000)]).astype(np.float32)
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode(x), t)


def test_quantize_divides_in_float32_like_torch():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, 50000).astype(np.float32)
    s = np.float32(np.max(np.abs(x)) / np.float32(448.0))
    ref = (torch.from_numpy(x) / torch.tensor(s, dtype=torch.float32)).to(torch.float8_e4m3fn)
    assert np.array_equal(e4m3.quantize(x, s), ref.view(torch.uint8).numpy())
    # the largest |x| lands on (or next to) the top code
    assert np.max(np.abs(e4m3.decode(e4m3.quantize(x, s)))) == 448.0


def test_dequantize_is_exact_product():
    s = np.float32(0.0123)
    codes = ALL[~np.isnan(e4m3.decode(ALL))]
    assert np.array_equal(e4m3.dequantize(codes, s), e4m3.decode(codes) * float(s))


def test_quantize_rejects_bad_scale():
    with pytest.raises(ValueError):
        e4m3.quantize([1.0], 0.0)
