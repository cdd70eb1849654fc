"""Seeded synthetic inputs (random numbers only; none of the method's arithmetic).

Both sides of every parity check draw their inputs from here: the CUDA path and
the oracle receive the same fp32 arrays.  The generator itself is in
``kvs_synth.c`` (SplitMix64 used counter-style + Box-Muller); this module
compiles it on first use and wraps it with numpy.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvs_synth.c")
_LIB = os.path.join(_HERE, "_build", "libkvs_synth.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``kvs_synth.c`` into ``_build/libkvs_synth.so`` (if stale) and return its path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, p = ctypes.c_uint64, ctypes.c_void_p
            lib.synth_u64.argtypes = [u64, u64, u64, u64, p]
            lib.synth_normal_f32.argtypes = [u64, u64, u64, u64, p]
            lib.synth_uniform_f32.argtypes = [u64, u64, u64, u64, ctypes.c_double, ctypes.c_double, p]
            for f in (lib.synth_u64, lib.synth_normal_f32, lib.synth_uniform_f32):
                f.restype = None
            _lib = lib
    return _lib


def tag(name: str, *ints: int) -> int:
    """A 64-bit stream tag from a name and integers (FNV-1a over the bytes)."""
    h = 0xCBF29CE484222325
    data = name.encode() + b"".join(int(i).to_bytes(8, "little", signed=True) for i in ints)
    for b in data:
        h = ((h ^ b) * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.uint64)
    if n:
        _load().synth_u64(seed, stream, offset, n, out.ctypes.data)
    return out


def normal(seed: int, stream: int, shape, offset: int = 0, out: np.ndarray | None = None) -> np.ndarray:
    """N(0,1) fp32 array of ``shape``: elements ``offset..`` of stream (seed, stream)."""
    shape = (shape,) if isinstance(shape, int) else tuple(shape)
    n = int(np.prod(shape)) if shape else 1
    if out is None:
        out = np.empty(shape, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous and out.size == n
    if n:
        _load().synth_normal_f32(seed, stream, offset, n, out.ctypes.data)
    return out


def uniform(seed: int, stream: int, shape, lo: float = 0.0, hi: float = 1.0, offset: int = 0) -> np.ndarray:
    shape = (shape,) if isinstance(shape, int) else tuple(shape)
    out = np.empty(shape, dtype=np.float32)
    if out.size:
        _load().synth_uniform_f32(seed, stream, offset, out.size, lo, hi, out.ctypes.data)
    return out


def choose(seed: int, stream: int, n: int, k: int, exclude=()) -> np.ndarray:
    """k distinct indices from range(n) minus ``exclude``, sorted (partial Fisher-Yates)."""
    pool = np.array([i for i in range(n) if i not in set(exclude)], dtype=np.int64)
    assert 0 <= k <= len(pool)
    r = u64(seed, stream, k)
    for i in range(k):
        j = i + int(r[i] % np.uint64(len(pool) - i))
        pool[i], pool[j] = pool[j], pool[i]
    return np.sort(pool[:k])
