"""kvs oracle -- TEST INFRASTRUCTURE ONLY.

Plain fp64 CPU model of streamed paged Q8_0-K / Q4_0-V attention (see the
header of ``kvs_oracle.c`` for the passages each function follows).  Only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvs_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libkvs_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``_build/libkvs_oracle.so`` (if stale) and return its path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.kvs_oracle_f32_to_f16.argtypes = [ctypes.c_float]
            lib.kvs_oracle_f32_to_f16.restype = ctypes.c_uint16
            lib.kvs_oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
            lib.kvs_oracle_f16_to_f32.restype = ctypes.c_float
            lib.kvs_oracle_q8_0_block.argtypes = [p, p, p]
            lib.kvs_oracle_q8_0_block.restype = None
            lib.kvs_oracle_q4_0_block.argtypes = [p, p, p]
            lib.kvs_oracle_q4_0_block.restype = None
            lib.kvs_oracle_quantize_kv.argtypes = [i64, i32, i32, p, p, p, p, p, p]
            lib.kvs_oracle_quantize_kv.restype = None
            lib.kvs_oracle_encode_page.argtypes = [i32, i32, i32, i64, i64, p, p, p, p, p]
            lib.kvs_oracle_encode_page.restype = None
            lib.kvs_oracle_attend.argtypes = [i64, i32, i32, p, p, p, p, i32, i32, p, i64, f64, p, p, i32]
            lib.kvs_oracle_attend.restype = i32
            lib.kvs_oracle_attend_partial.argtypes = [i64, i32, i32, p, p, p, p, i32, i32, p, i64, f64,
                                                      i64, i64, p, p, p]
            lib.kvs_oracle_attend_partial.restype = i32
            lib.kvs_oracle_combine.argtypes = [i32, i32, p, p, p, p, p]
            lib.kvs_oracle_combine.restype = None
            lib.kvs_oracle_f32_to_f16_n.argtypes = [i64, p, p]
            lib.kvs_oracle_f32_to_f16_n.restype = None
            lib.kvs_oracle_f16_to_f32_n.argtypes = [i64, p, p]
            lib.kvs_oracle_f16_to_f32_n.restype = None
            lib.kvs_oracle_threads.argtypes = [i32]
            lib.kvs_oracle_threads.restype = i32
            _lib = lib
    return _lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- fp16

def f32_to_f16_bits(x) -> np.ndarray:
    """IEEE binary16 bits (round to nearest even) of each fp32 value."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().kvs_oracle_f32_to_f16_n(x.size, x.ctypes.data, out.ctypes.data)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().kvs_oracle_f16_to_f32_n(h.size, h.ctypes.data, out.ctypes.data)
    return out


# ---------------------------------------------------------- quantisers

def q8_0_block(x):
    """One Q8_0 block: (int8 codes[32], fp16 scale bits)."""
    x = _c(x, np.float32)
    assert x.shape == (32,)
    q = np.zeros(32, dtype=np.int8)
    d = np.zeros(1, dtype=np.uint16)
    _load().kvs_oracle_q8_0_block(x.ctypes.data, q.ctypes.data, d.ctypes.data)
    return q, int(d[0])


def q4_0_block(x):
    """One Q4_0 block: (codes 0..15 [32] unpacked, fp16 scale bits)."""
    x = _c(x, np.float32)
    assert x.shape == (32,)
    q = np.zeros(32, dtype=np.uint8)
    d = np.zeros(1, dtype=np.uint16)
    _load().kvs_oracle_q4_0_block(x.ctypes.data, q.ctypes.data, d.ctypes.data)
    return q, int(d[0])


class QuantKV:
    """Quantised history: kq int8 [T][Hk][D], kd u16 [T][Hk][D/32], vq u8 [T][Hk][D], vd u16."""

    def __init__(self, k: np.ndarray, v: np.ndarray):
        k = _c(k, np.float32)
        v = _c(v, np.float32)
        assert k.shape == v.shape and k.ndim == 3 and k.shape[2] % 32 == 0
        self.T, self.Hk, self.D = k.shape
        nb = self.D // 32
        self.kq = np.empty(k.shape, dtype=np.int8)
        self.kd = np.empty((self.T, self.Hk, nb), dtype=np.uint16)
        self.vq = np.empty(k.shape, dtype=np.uint8)
        self.vd = np.empty((self.T, self.Hk, nb), dtype=np.uint16)
        if self.T:
            _load().kvs_oracle_quantize_kv(self.T, self.Hk, self.D, k.ctypes.data, v.ctypes.data,
                                           self.kq.ctypes.data, self.kd.ctypes.data,
                                           self.vq.ctypes.data, self.vd.ctypes.data)

    def _ptrs(self):
        return (self.kq.ctypes.data, self.kd.ctypes.data, self.vq.ctypes.data, self.vd.ctypes.data)

    def encode_page(self, P: int, page: int) -> np.ndarray:
        out = np.empty(P * self.Hk * self.D * 13 // 8, dtype=np.uint8)
        _load().kvs_oracle_encode_page(P, self.Hk, self.D, self.T, page, *self._ptrs(),
                                       out.ctypes.data)
        return out

    def attend(self, q: np.ndarray, pos0: int, scale: float, threads: int = 0):
        """Causal attention of q [R][Hq][D] at positions pos0..: (o fp64 [R][Hq][D], lse [R][Hq])."""
        q = _c(q, np.float32)
        R, Hq, D = q.shape
        assert D == self.D
        o = np.empty((R, Hq, D), dtype=np.float64)
        lse = np.empty((R, Hq), dtype=np.float64)
        rc = _load().kvs_oracle_attend(self.T, self.Hk, D, *self._ptrs(), R, Hq, q.ctypes.data,
                                       pos0, scale, o.ctypes.data, lse.ctypes.data, threads)
        if rc != 0:
            raise ValueError("kvs_oracle_attend: invalid arguments")
        return o, lse

    def attend_partial(self, q: np.ndarray, pos0: int, scale: float, k0: int, k1: int):
        """(m [R][Hq], l [R][Hq], o_unnormalised [R][Hq][D]) over keys [k0, k1)."""
        q = _c(q, np.float32)
        R, Hq, D = q.shape
        m = np.empty((R, Hq), dtype=np.float64)
        l = np.empty((R, Hq), dtype=np.float64)
        o = np.empty((R, Hq, D), dtype=np.float64)
        rc = _load().kvs_oracle_attend_partial(self.T, self.Hk, D, *self._ptrs(), R, Hq,
                                               q.ctypes.data, pos0, scale, k0, k1, m.ctypes.data,
                                               l.ctypes.data, o.ctypes.data)
        if rc != 0:
            raise ValueError("kvs_oracle_attend_partial: invalid arguments")
        return m, l, o


def combine(m, l, o_part):
    """Log-sum-exp combine of partials of one (row, head): m, l [S]; o_part [S][D]."""
    m = _c(m, np.float64)
    l = _c(l, np.float64)
    o_part = _c(o_part, np.float64)
    S, D = o_part.shape
    o = np.empty(D, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    _load().kvs_oracle_combine(S, D, m.ctypes.data, l.ctypes.data, o_part.ctypes.data,
                               o.ctypes.data, lse.ctypes.data)
    return o, float(lse[0])


def threads(n: int = 0) -> int:
    """Threads ``attend(..., threads=n)`` uses."""
    return int(_load().kvs_oracle_threads(n))
