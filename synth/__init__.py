"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This package holds no attention, cache or allocator arithmetic: it only
draws numbers (normal deviates, integers, permutations) and lays out the
workloads' shapes.  ``gen.c`` does the bulk normal draws (counter-based, so
any sub-range can be drawn on its own); the integer draws use the same
SplitMix64 finaliser in numpy.
"""

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_SRC = os.path.join(_HERE, "gen.c")
_lock = threading.Lock()
_lib = None

GOLDEN = np.uint64(0x9E3779B97F4A7C15)


def build(force=False):
    """Compile ``gen.c`` into ``_synth.so`` next to it (gcc, OpenMP)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_SO)
            u64, i64 = ctypes.c_uint64, ctypes.c_int64
            vp = ctypes.c_void_p
            lib.synth_key.argtypes = [u64, u64]
            lib.synth_key.restype = u64
            for name in ("synth_normal_f32", "synth_normal_f64", "synth_u64"):
                getattr(lib, name).argtypes = [u64, u64, u64, i64, vp]
                getattr(lib, name).restype = None
            _lib = lib
    return _lib


def normal_f32(seed, stream, n, offset=0):
    """``n`` float32 normal deviates of stream ``stream`` starting at ``offset``."""
    out = np.empty(int(n), dtype=np.float32)
    if n:
        _load().synth_normal_f32(seed, stream, offset, int(n), out.ctypes.data)
    return out


def normal_f64(seed, stream, n, offset=0):
    out = np.empty(int(n), dtype=np.float64)
    if n:
        _load().synth_normal_f64(seed, stream, offset, int(n), out.ctypes.data)
    return out


def u64(seed, stream, n, offset=0):
    """``n`` raw 64-bit draws of a stream."""
    out = np.empty(int(n), dtype=np.uint64)
    if n:
        _load().synth_u64(seed, stream, offset, int(n), out.ctypes.data)
    return out


def uniform_int(seed, stream, n, lo, hi):
    """``n`` integers uniform in ``[lo, hi]`` (inclusive), by ``draw mod range``."""
    r = np.uint64(hi - lo + 1)
    return (u64(seed, stream, n) % r).astype(np.int64) + lo


def permutation(seed, stream, n):
    """A seeded permutation of ``0..n-1``: the stable argsort of ``n`` draws."""
    return np.argsort(u64(seed, stream, n), kind="stable").astype(np.int64)


def sample_without_replacement(seed, stream, population, k):
    """``k`` distinct elements of ``population`` (an int array), seeded."""
    population = np.asarray(population)
    if k > len(population):
        raise ValueError("sample larger than population")
    return population[permutation(seed, stream, len(population))[:k]]
