"""Build and call the C binary64 decode oracle (``decode_ref.c``).

Test infrastructure only (see ``oracle/__init__``). Compiled with gcc + OpenMP into
``oracle/_build/liboracle.so``; shares nothing with the CUDA library.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "decode_ref.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc -O2 -fopenmp); returns its path."""
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    if force or not os.path.exists(_OUT) or os.path.getmtime(_OUT) < os.path.getmtime(_SRC):
        subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", _OUT, _SRC, "-lm"],
                       check=True)
    return _OUT


def _load():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        f = _lib.oracle_decode
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                      ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                      ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
        f2 = _lib.oracle_prefill
        f2.restype = ctypes.c_int
        f2.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                       ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                       ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                       ctypes.c_int]
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float64:
        return 3
    raise TypeError(f"oracle stores float32 or bf16 bits (uint16), got {a.dtype}")


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, tables: np.ndarray,
           lens: np.ndarray, scale: float, rows: Optional[Sequence[int]] = None,
           n_threads: int = 0, return_threads: bool = False, window: int = 0):
    """Binary64 paged decode. q [n, Hq, D]; caches [NB, Hkv, B, D]; tables [n, MB].
    window > 0: attend only to the last ``window`` positions of each sequence.

    Returns out [n, Hq, D] (rows=None) or [len(rows), D] for flat (b * Hq + j) ids.
    """
    lib = _load()
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    n, Hq, D = q.shape
    _, Hkv, B, D2 = k_cache.shape
    assert D2 == D and v_cache.shape == k_cache.shape and k_cache.dtype == v_cache.dtype
    rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n_rows = n * Hq if rows_arr is None else rows_arr.size
    out = np.zeros((n_rows, D), dtype=np.float64)
    used = lib.oracle_decode(out.ctypes.data, q.ctypes.data, _dtype_code(q), k_cache.ctypes.data,
                             v_cache.ctypes.data, _dtype_code(k_cache), tables.ctypes.data, lens.ctypes.data,
                             n, Hq, Hkv, D, B, tables.shape[1], float(scale), int(window),
                             None if rows_arr is None else rows_arr.ctypes.data, n_rows, int(n_threads))
    if used < 0:
        raise ValueError("oracle_decode rejected its arguments")
    res = out.reshape(n, Hq, D) if rows_arr is None else out
    return (res, used) if return_threads else res


def prefill(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, tables: np.ndarray, lens: np.ndarray,
            cu_q: np.ndarray, scale: float, window: int = 0, n_threads: int = 0) -> np.ndarray:
    """Binary64 causal prefill over pages (see oracle_prefill in decode_ref.c). q [total_q, Hq, D]."""
    lib = _load()
    q = np.ascontiguousarray(q)
    k_cache = np.ascontiguousarray(k_cache)
    v_cache = np.ascontiguousarray(v_cache)
    tables = np.ascontiguousarray(tables, dtype=np.int32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    cu_q = np.ascontiguousarray(cu_q, dtype=np.int32)
    total, Hq, D = q.shape
    _, Hkv, B, _ = k_cache.shape
    out = np.zeros((total, Hq, D), dtype=np.float64)
    used = lib.oracle_prefill(out.ctypes.data, q.ctypes.data, _dtype_code(q), k_cache.ctypes.data,
                              v_cache.ctypes.data, _dtype_code(k_cache), tables.ctypes.data, lens.ctypes.data,
                              cu_q.ctypes.data, lens.size, Hq, Hkv, D, B, tables.shape[1], float(scale), int(window),
                              int(n_threads))
    if used < 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return out


def decode_fn_from(lib_path: str):
    """A ``decode``-like callable bound to another build of ``decode_ref.c`` (used to test the pins)."""
    lib = ctypes.CDLL(lib_path)
    f = lib.oracle_decode
    f.restype = ctypes.c_int
    f.argtypes = _load().oracle_decode.argtypes

    def run(q, k_cache, v_cache, tables, lens, scale, window=0):
        q = np.ascontiguousarray(q)
        k_cache = np.ascontiguousarray(k_cache)
        v_cache = np.ascontiguousarray(v_cache)
        tables = np.ascontiguousarray(tables, dtype=np.int32)
        lens = np.ascontiguousarray(lens, dtype=np.int32)
        n, Hq, D = q.shape
        _, Hkv, B, _ = k_cache.shape
        out = np.zeros((n * Hq, D), dtype=np.float64)
        f(out.ctypes.data, q.ctypes.data, _dtype_code(q), k_cache.ctypes.data, v_cache.ctypes.data,
          _dtype_code(k_cache), tables.ctypes.data, lens.ctypes.data, n, Hq, Hkv, D, B, tables.shape[1],
          float(scale), int(window), None, n * Hq, 1)
        return out.reshape(n, Hq, D)
    return run
