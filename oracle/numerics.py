"""Exact conversions between the cache element types and float64.

Test infrastructure only (see ``oracle/__init__.py``).

The cache model keeps each element type as numpy data with exactly the
stored bits:

* ``f32``      numpy float32
* ``f16``      numpy float16 (IEEE binary16)
* ``bf16``     numpy uint16 holding bfloat16 bit patterns (the upper half of
               a float32)
* ``fp8_e4m3`` numpy uint8 holding E4M3 codes (see ``oracle.e4m3``)

Widening any of them to float64 is exact.  Narrowing float32 to f16 / bf16
rounds to nearest, ties to even.
"""

import numpy as np

from . import e4m3

KV_DTYPES = ("f32", "f16", "bf16", "fp8_e4m3")
STORAGE = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "fp8_e4m3": np.uint8}


def bf16_bits_to_f64(bits):
    """Value of bfloat16 bit patterns: they are the top 16 bits of a float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x):
    """bfloat16 bits of float32 values, rounded to nearest, ties to even.

    The 16 dropped bits decide the rounding: above half an ulp rounds up,
    exactly half rounds to the even result.  NaN stays a quiet NaN.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    hi = u >> np.uint64(16)
    lo = u & np.uint64(0xFFFF)
    up = (lo > 0x8000) | ((lo == 0x8000) & ((hi & np.uint64(1)) == 1))
    r = hi + up.astype(np.uint64)
    isnan = np.isnan(np.asarray(x, dtype=np.float32))
    r = np.where(isnan, (hi | np.uint64(0x40)) & np.uint64(0xFFFF), r)
    return r.astype(np.uint16)


def to_f64(data, dtype, scale=1.0):
    """Exact float64 value of stored cache elements of type ``dtype``.

    For ``fp8_e4m3`` the value is the dequantised ``decode(code) * scale``.
    """
    if dtype == "f32":
        return np.asarray(data, dtype=np.float32).astype(np.float64)
    if dtype == "f16":
        return np.asarray(data, dtype=np.float16).astype(np.float64)
    if dtype == "bf16":
        return bf16_bits_to_f64(data)
    if dtype == "fp8_e4m3":
        return e4m3.dequantize(data, scale)
    raise ValueError(f"unknown dtype {dtype!r}")


def source_to_f32(data, dtype):
    """Float32 value of a source (new K/V token) array of type f32/f16/bf16."""
    if dtype == "f32":
        return np.asarray(data, dtype=np.float32)
    if dtype == "f16":
        return np.asarray(data, dtype=np.float16).astype(np.float32)
    if dtype == "bf16":
        return bf16_bits_to_f64(data).astype(np.float32)
    raise ValueError(f"unsupported source dtype {dtype!r}")


def store(src, src_dtype, cache_dtype, scale=1.0):
    """Bits the cache holds for source values ``src`` of type ``src_dtype``.

    Same type: the bits are copied.  float32 into f16 / bf16: rounded to
    nearest even.  Anything into fp8_e4m3: ``e4m3.quantize`` with ``scale``.
    Other combinations are not part of the path and raise ValueError.
    """
    if cache_dtype == "fp8_e4m3":
        return e4m3.quantize(source_to_f32(src, src_dtype), scale)
    if src_dtype == cache_dtype:
        return np.asarray(src, dtype=STORAGE[cache_dtype]).copy()
    if src_dtype == "f32" and cache_dtype == "f16":
        return np.asarray(src, dtype=np.float32).astype(np.float16)
    if src_dtype == "f32" and cache_dtype == "bf16":
        return f32_to_bf16_bits(src)
    raise ValueError(f"append {src_dtype} -> {cache_dtype} is not supported")
