"""All-core OpenMP CPU baseline of one tree level (a measured comparison point for the benchmark).

A feature-parallel histogram fill, sibling subtraction and a serial split scan in ``omp_level.c``,
independent of both the CUDA library and the oracle. ``build()`` compiles it with gcc and OpenMP;
``level()`` runs one level on numpy inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "omp_level.c")
_LIB = os.path.join(_HERE, "_build", "libomp_level.so")
_lock = threading.Lock()
_lib = None

SPLIT_DTYPE = np.dtype([
    ("feature", "<i4"), ("bin", "<i4"), ("default_left", "u1"), ("pad", "u1", (7,)), ("gain", "<f8"),
    ("g_left", "<i8"), ("h_left", "<i8"), ("g_right", "<i8"), ("h_right", "<i8"),
])


def build(force: bool = False) -> str:
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-o", tmp,
                        _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        p, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        L.omp_level.argtypes = [p, ctypes.c_int, i64, i32, i32, ctypes.c_uint32, p, p, p, i32, p, p, p,
                                f64, f64, f64, f64, f64, p, p]
        L.omp_level.restype = ctypes.c_int
        L.omp_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def threads() -> int:
    return int(lib().omp_threads())


def quantise(gpair, scale_g, scale_h):
    """The quantised pairs the baseline fills with: round-half-even of the float32 product, int32 [N][2]
    (inputs must keep |x * s| < 2^31)."""
    gp = np.ascontiguousarray(gpair, dtype=np.float32).reshape(-1, 2)
    prod = gp * np.array([scale_g, scale_h], dtype=np.float32)
    if not np.all(np.abs(prod) < 2.0 ** 31):
        raise ValueError("quantised value out of the int32 range")
    return np.rint(prod).astype(np.int32)


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def level(bins, n_bins, sentinel, q, rows, offsets, parent=None, lam=1.0, gamma=0.0, mcw=0.0, scale_g=1.0,
          scale_h=1.0):
    """One level: returns (small_hist, large_hist or None, small_splits, large_splits or None).
    bins feature-major [F][N]; q int32 [N][2] quantised pairs; rows int32 or None; offsets int64 [n+1];
    parent int64 [n][F][B][2] or None."""
    bins = np.ascontiguousarray(bins)
    F, N = bins.shape
    q = np.ascontiguousarray(q, dtype=np.int32)
    offs = np.ascontiguousarray(offsets, dtype=np.int64)
    n = offs.shape[0] - 1
    rows = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    small = np.empty((n, F, n_bins + 1, 2), np.int64)
    large = np.empty_like(small) if parent is not None else None
    par = None if parent is None else np.ascontiguousarray(parent, dtype=np.int64)
    so = np.zeros(n, SPLIT_DTYPE)
    lo = np.zeros(n, SPLIT_DTYPE) if parent is not None else None
    st = lib().omp_level(_p(bins), bins.dtype.itemsize, N, F, n_bins, sentinel, _p(q), _p(rows), _p(offs), n,
                         _p(par), _p(small), _p(large), float(lam), float(gamma), float(mcw),
                         1.0 / float(np.float32(scale_g)), 1.0 / float(np.float32(scale_h)), _p(so), _p(lo))
    if st != 0:
        raise ValueError("omp_level: bad arguments")
    return small, large, so, lo
