"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle's callers.

The module holds none of the decode step's arithmetic: it turns (seed, stream,
index) into numbers through the counter-based generator in ``grgen.c`` and
lays the numbers out as the workloads ask.  Every value is a pure function of
(seed, stream, index), so any slice of any tensor can be regenerated alone.

bf16 tensors are returned as ``numpy.uint16`` arrays holding the bf16 bit
patterns; float32 tensors as ``numpy.float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "grgen.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libgrgen.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile grgen.c into gen/_build/libgrgen.so (gcc, OpenMP, no FP contraction)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-shared",
                           "-fPIC", "-o", tmp, _SRC])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int32
            lib.grgen_word.restype = u64
            lib.grgen_word.argtypes = [u64, u64, u64]
            lib.grgen_quantile.restype = ctypes.c_double
            lib.grgen_quantile.argtypes = [ctypes.c_int]
            lib.grgen_normal.restype = None
            lib.grgen_normal.argtypes = [u64, u64, ctypes.c_double, ctypes.c_double, ctypes.c_int,
                                         ctypes.c_void_p, i64, i64]
            lib.grgen_ints.restype = None
            lib.grgen_ints.argtypes = [u64, u64, i32, i32, ctypes.c_void_p, i64, i64]
            lib.grgen_permutation.restype = None
            lib.grgen_permutation.argtypes = [u64, u64, ctypes.c_void_p, i64]
            _lib = lib
    return _lib


def word(seed: int, stream: int, i: int) -> int:
    return _load().grgen_word(seed, stream, i)


def quantile(k: int) -> float:
    return _load().grgen_quantile(k)


def normal(seed: int, stream: int, shape, sigma: float = 1.0, mean: float = 0.0,
           dtype: str = "bf16", offset: int = 0) -> np.ndarray:
    """Array of N(mean, sigma^2) draws; element i (C order) uses counter offset + i."""
    n = int(np.prod(shape))
    if dtype == "bf16":
        out = np.empty(n, dtype=np.uint16)
        code = 1
    elif dtype == "f32":
        out = np.empty(n, dtype=np.float32)
        code = 0
    else:
        raise ValueError(dtype)
    if n:
        _load().grgen_normal(seed, stream, float(mean), float(sigma), code,
                             out.ctypes.data, n, int(offset))
    return out.reshape(shape)


def ints(seed: int, stream: int, lo: int, hi: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().grgen_ints(seed, stream, lo, hi, out.ctypes.data, n, offset)
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    if n:
        _load().grgen_permutation(seed, stream, out.ctypes.data, n)
    return out


def bf16_bits_to_f32(a: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to float32."""
    return (a.astype(np.uint32) << 16).view(np.float32)


from .workloads import (Workload, WORKLOADS, ModelWeights, make_weights, prompt_tokens,  # noqa: E402
                        kv_prefill, slot_map, row_positions, STREAM)

__all__ = ["build", "word", "quantile", "normal", "ints", "permutation", "bf16_bits_to_f32",
           "Workload", "WORKLOADS", "ModelWeights", "make_weights", "prompt_tokens", "kv_prefill",
           "slot_map", "row_positions", "STREAM"]
