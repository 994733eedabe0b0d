"""FP8 E4M3 codec for the quantised KV cache.

Test infrastructure only (see ``oracle/__init__.py``).

[DEV] section 6 item 4 "Enable FP8 KV Cache" and [HI] "KV quantization cuts
memory in half" store K and V in one byte instead of two but do not fix the
8-bit format.  Reading taken: the OCP 8-bit floating point "E4M3" encoding
(the variant without infinities, often called E4M3FN):

* bit 7 sign, bits 6..3 exponent field E (bias 7), bits 2..0 mantissa M;
* E == 0          : subnormal, value = (-1)^s * 2^-6 * M/8;
* 1 <= E <= 15    : normal, value = (-1)^s * 2^(E-7) * (1 + M/8);
* E == 15, M == 7 : NaN (0x7F / 0xFF); there is no infinity;
* largest finite magnitude 2^8 * 1.75 = 448, smallest 2^-9.

Encoding rounds to nearest with ties to the even code and saturates every
finite magnitude beyond 448 to 448.  The cache stores ``encode(x / scale)``
with the division done in IEEE float32, and the dequantised value is
``decode(code) * scale`` (one float32 scale per cache tensor).
"""

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_MIN_SUBNORMAL = 2.0 ** -9
E4M3_NAN_CODE = 0x7F


def decode(codes):
    """Value of each E4M3 code, from the bit fields (float64; NaN codes -> nan)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    sub = np.ldexp(m / 8.0, -6)
    nor = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    mag = np.where(e == 0, sub, nor)
    mag = np.where((e == 15) & ((c & 7) == 7), np.nan, mag)
    return sign * mag


def encode(x):
    """E4M3 code of each value: round to nearest, ties to even, saturate to 448.

    ``x`` is taken exactly (any float dtype; the float32 quotient the cache
    stores is exact in float64).  NaN encodes as 0x7F.  The sign of zero and
    of values that round to zero is kept (code 0x80 for negative ones).
    """
    x = np.asarray(x, dtype=np.float64)
    neg = np.signbit(x)
    a = np.abs(x)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, a)
    sat = a >= E4M3_MAX
    a = np.where(sat, 0.0, a)
    # spacing of representable values around a: 2^-9 below the smallest
    # normal, otherwise 2^(e-3) for a in [2^e, 2^(e+1)) (3 mantissa bits)
    _, exp2 = np.frexp(a)          # a = f * 2^exp2, f in [0.5, 1)
    e = exp2.astype(np.int64) - 1  # a in [2^e, 2^(e+1))
    quantum_exp = np.where(a < E4M3_MIN_NORMAL, -9, e - 3)
    n = np.rint(np.ldexp(a, -quantum_exp))          # RNE on an exact scaling
    value = np.ldexp(n, quantum_exp)                  # representable magnitude
    value = np.where(sat, E4M3_MAX, value)
    # bit fields of the representable magnitude
    is_sub = value < E4M3_MIN_NORMAL
    sub_m = np.rint(np.ldexp(value, 9)).astype(np.int64)   # 0..7 (8 == min normal)
    _, vexp = np.frexp(np.where(is_sub, 1.0, value))
    ve = vexp.astype(np.int64) - 1
    vm = np.rint((np.ldexp(np.where(is_sub, 1.0, value), -ve) - 1.0) * 8.0).astype(np.int64)
    nor_code = ((ve + 7) << 3) | vm
    code = np.where(is_sub, sub_m, nor_code)
    code = np.where(neg, code | 0x80, code)
    code = np.where(nan, E4M3_NAN_CODE, code)
    return code.astype(np.uint8)


def quantize(x_f32, scale_f32):
    """Cache code for each source value: ``encode(float32(x) / float32(scale))``.

    The quotient is the IEEE float32 division of the float32 source value by
    the float32 scale; the encoder then rounds that exact float32 value.
    """
    xs = np.asarray(x_f32, dtype=np.float32)
    s = np.float32(scale_f32)
    if not (np.isfinite(s) and s > 0):
        raise ValueError("FP8 scale must be a finite positive float32")
    with np.errstate(over="ignore"):
        q = (xs / s).astype(np.float32)
    return encode(q)


def dequantize(codes, scale_f32):
    """Dequantised value of each cache code, exact in float64: decode * scale."""
    return decode(codes) * float(np.float32(scale_f32))
