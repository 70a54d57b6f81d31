"""CPU oracle for the level histogram path: ctypes wrapper around ``gbt_oracle.c``.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the CUDA library and its
Python binding never do. It shares no code with them.

``build()`` compiles ``gbt_oracle.c`` with gcc (``-O2 -ffp-contract=off``) into
``oracle/_build/libgbt_oracle.so``. The functions below take and return numpy
arrays; each cites the passage it follows in ``gbt_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gbt_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libgbt_oracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_BIN, ERR_ROW, ERR_QUANT, ERR_INCONSISTENT = range(6)


class Split(ctypes.Structure):
    _fields_ = [
        ("feature", ctypes.c_int32),
        ("bin", ctypes.c_int32),
        ("default_left", ctypes.c_uint8),
        ("pad", ctypes.c_uint8 * 7),
        ("gain", ctypes.c_double),
        ("g_left", ctypes.c_int64),
        ("h_left", ctypes.c_int64),
        ("g_right", ctypes.c_int64),
        ("h_right", ctypes.c_int64),
    ]


SPLIT_DTYPE = np.dtype(
    [
        ("feature", "<i4"),
        ("bin", "<i4"),
        ("default_left", "u1"),
        ("pad", "u1", (7,)),
        ("gain", "<f8"),
        ("g_left", "<i8"),
        ("h_left", "<i8"),
        ("g_right", "<i8"),
        ("h_right", "<i8"),
    ]
)
assert SPLIT_DTYPE.itemsize == ctypes.sizeof(Split) == 56


def build(force: bool = False) -> str:
    """Compile the oracle with gcc; returns the shared-library path."""
    with _lock:
        if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
            return _LIB_PATH
        os.makedirs(_OUT_DIR, exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-Wall", "-Wextra", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        L.oracle_quantise.argtypes = [p, i64, f32, f32, p]
        L.oracle_quantise.restype = ctypes.c_int
        L.oracle_max_abs_q.argtypes = [p, i64]
        L.oracle_max_abs_q.restype = i64
        L.oracle_build_hist.argtypes = [p, ctypes.c_int, i64, i32, i32, ctypes.c_uint32, p, p, p, i32, p]
        L.oracle_build_hist.restype = ctypes.c_int
        L.oracle_build_hist_multi.argtypes = [p, ctypes.c_int, i64, i32, i32, ctypes.c_uint32, p, i32, p, p, i32, p]
        L.oracle_build_hist_multi.restype = ctypes.c_int
        L.oracle_subtract.argtypes = [p, p, p, p, i32, i32, i32]
        L.oracle_subtract.restype = ctypes.c_int
        L.oracle_gain.argtypes = [f64] * 8
        L.oracle_gain.restype = f64
        L.oracle_find_splits.argtypes = [p, i32, i32, i32, f64, f64, f64, f64, f64, p]
        L.oracle_find_splits.restype = ctypes.c_int
        L.oracle_find_level_split.argtypes = [p, i32, i32, i32, f64, f64, f64, f64, f64, p]
        L.oracle_find_level_split.restype = ctypes.c_int
        L.oracle_build_hist_f64.argtypes = [p, ctypes.c_int, i64, i32, i32, ctypes.c_uint32, p, p, p, i32, p, p]
        L.oracle_build_hist_f64.restype = ctypes.c_int
        L.oracle_subtract_f64.argtypes = [p, p, p, p, i32, i32, i32]
        L.oracle_subtract_f64.restype = ctypes.c_int
        L.oracle_find_splits_f64.argtypes = [p, i32, i32, i32, f64, f64, f64, p]
        L.oracle_find_splits_f64.restype = ctypes.c_int
        L.oracle_partition.argtypes = [p, ctypes.c_int, i64, i32, ctypes.c_uint32, p, p, i32, p, p, p]
        L.oracle_partition.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def quantise(gpair: np.ndarray, scale_g: float, scale_h: float):
    """[n][2] float32 -> ([n][2] int32, status). Rounding: float32 product, then round-half-even."""
    gp = np.ascontiguousarray(gpair, dtype=np.float32).reshape(-1, 2)
    q = np.empty_like(gp, dtype=np.int32)
    st = lib().oracle_quantise(_ptr(gp), gp.shape[0], float(scale_g), float(scale_h), _ptr(q))
    return q, st


def max_abs_q(q: np.ndarray) -> int:
    q = np.ascontiguousarray(q, dtype=np.int32)
    return int(lib().oracle_max_abs_q(_ptr(q), q.shape[0]))


def build_hist(bins: np.ndarray, n_bins: int, sentinel: int, q: np.ndarray, rows, node_offsets):
    """bins feature-major [F][N] (uint8/uint16); returns (hist [n_nodes][F][n_bins+1][2] int64, status)."""
    bins = np.ascontiguousarray(bins)
    assert bins.dtype in (np.uint8, np.uint16) and bins.ndim == 2
    F, N = bins.shape
    q = np.ascontiguousarray(q, dtype=np.int32).reshape(-1, 2)
    assert q.shape[0] == N
    offs = np.ascontiguousarray(node_offsets, dtype=np.int64)
    n_nodes = offs.shape[0] - 1
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    hist = np.empty((n_nodes, F, n_bins + 1, 2), dtype=np.int64)
    st = lib().oracle_build_hist(_ptr(bins), bins.dtype.itemsize, N, F, n_bins, sentinel, _ptr(q), _ptr(rows_a),
                                 _ptr(offs), n_nodes, _ptr(hist))
    return hist, st


def quantise_multi(gpair: np.ndarray, scales_g, scales_h):
    """gpair float32 [N][k][2], one scale pair per target -> (q int32 [N][k][2], status): each target's pairs
    quantised with its own scales."""
    gp = np.ascontiguousarray(gpair, dtype=np.float32)
    N, k, _ = gp.shape
    q = np.empty((N, k, 2), dtype=np.int32)
    st = OK
    for t in range(k):
        qt, s = quantise(gp[:, t, :], scales_g[t], scales_h[t])
        q[:, t, :] = qt.reshape(N, 2)
        st = st if st != OK else s
    return q, st


def build_hist_multi(bins: np.ndarray, n_bins: int, sentinel: int, q: np.ndarray, rows, node_offsets):
    """Multi-output histograms: q int32 [N][k][2] -> (hist [k][n_nodes][F][n_bins+1][2] int64, status)."""
    bins = np.ascontiguousarray(bins)
    F, N = bins.shape
    q = np.ascontiguousarray(q, dtype=np.int32)
    assert q.ndim == 3 and q.shape[0] == N and q.shape[2] == 2
    k = q.shape[1]
    offs = np.ascontiguousarray(node_offsets, dtype=np.int64)
    n_nodes = offs.shape[0] - 1
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    hist = np.empty((k, n_nodes, F, n_bins + 1, 2), dtype=np.int64)
    st = lib().oracle_build_hist_multi(_ptr(bins), bins.dtype.itemsize, N, F, n_bins, sentinel, _ptr(q), k,
                                       _ptr(rows_a), _ptr(offs), n_nodes, _ptr(hist))
    return hist, st


def subtract(parent: np.ndarray, parent_of, small: np.ndarray):
    """large[p] = parent[parent_of[p]] - small[p]; returns (large, status)."""
    parent = np.ascontiguousarray(parent, dtype=np.int64)
    small = np.ascontiguousarray(small, dtype=np.int64)
    n_pairs, F, B, two = small.shape
    assert two == 2 and parent.shape[1:] == small.shape[1:]
    po = None if parent_of is None else np.ascontiguousarray(parent_of, dtype=np.int32)
    large = np.empty_like(small)
    st = lib().oracle_subtract(_ptr(parent), _ptr(po), _ptr(small), _ptr(large), n_pairs, F, B)
    return large, st


def gain(gl, hl, gr, hr, g, h, lam, gamma) -> float:
    return float(lib().oracle_gain(gl, hl, gr, hr, g, h, lam, gamma))


def find_splits(hist: np.ndarray, n_bins: int, lam: float, gamma: float, min_child_weight: float,
                scale_g: float, scale_h: float):
    """hist [n_nodes][F][n_bins+1][2] int64 -> (structured array of SPLIT_DTYPE, status)."""
    hist = np.ascontiguousarray(hist, dtype=np.int64)
    n_nodes, F, B, _ = hist.shape
    assert B == n_bins + 1
    out = np.zeros(n_nodes, dtype=SPLIT_DTYPE)
    inv_sg = 1.0 / float(np.float32(scale_g))
    inv_sh = 1.0 / float(np.float32(scale_h))
    st = lib().oracle_find_splits(_ptr(hist), n_nodes, F, n_bins, lam, gamma, min_child_weight, inv_sg, inv_sh,
                                  _ptr(out))
    return out, st


def find_level_split(hist: np.ndarray, n_bins: int, lam: float, gamma: float, min_child_weight: float,
                     scale_g: float, scale_h: float):
    """Oblivious level split: hist [n_nodes][F][n_bins+1][2] int64 -> (one SPLIT_DTYPE record, status)."""
    hist = np.ascontiguousarray(hist, dtype=np.int64)
    n_nodes, F, B, _ = hist.shape
    assert B == n_bins + 1
    out = np.zeros(1, dtype=SPLIT_DTYPE)
    inv_sg = 1.0 / float(np.float32(scale_g))
    inv_sh = 1.0 / float(np.float32(scale_h))
    st = lib().oracle_find_level_split(_ptr(hist), n_nodes, F, n_bins, lam, gamma, min_child_weight, inv_sg, inv_sh,
                                       _ptr(out))
    return out[0], st


SPLIT_F64_DTYPE = np.dtype([
    ("feature", "<i4"), ("bin", "<i4"), ("default_left", "u1"), ("pad", "u1", (7,)), ("gain", "<f8"),
    ("g_left", "<f8"), ("h_left", "<f8"), ("g_right", "<f8"), ("h_right", "<f8"),
])


def build_hist_f64(bins: np.ndarray, n_bins: int, sentinel: int, gpair: np.ndarray, rows, node_offsets):
    """Float-cell mode: (hist, abs_hist, status), both [n_nodes][F][n_bins+1][2] float64; abs_hist holds the
    sums of |g|, |h| per cell."""
    bins = np.ascontiguousarray(bins)
    F, N = bins.shape
    gp = np.ascontiguousarray(gpair, dtype=np.float32).reshape(-1, 2)
    assert gp.shape[0] == N
    offs = np.ascontiguousarray(node_offsets, dtype=np.int64)
    n_nodes = offs.shape[0] - 1
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    hist = np.empty((n_nodes, F, n_bins + 1, 2), dtype=np.float64)
    ab = np.empty_like(hist)
    st = lib().oracle_build_hist_f64(_ptr(bins), bins.dtype.itemsize, N, F, n_bins, sentinel, _ptr(gp), _ptr(rows_a),
                                     _ptr(offs), n_nodes, _ptr(hist), _ptr(ab))
    return hist, ab, st


def subtract_f64(parent: np.ndarray, parent_of, small: np.ndarray):
    parent = np.ascontiguousarray(parent, dtype=np.float64)
    small = np.ascontiguousarray(small, dtype=np.float64)
    n_pairs, F, B, _ = small.shape
    po = None if parent_of is None else np.ascontiguousarray(parent_of, dtype=np.int32)
    large = np.empty_like(small)
    st = lib().oracle_subtract_f64(_ptr(parent), _ptr(po), _ptr(small), _ptr(large), n_pairs, F, B)
    return large, st


def find_splits_f64(hist: np.ndarray, n_bins: int, lam: float, gamma: float, min_child_weight: float):
    hist = np.ascontiguousarray(hist, dtype=np.float64)
    n_nodes, F, B, _ = hist.shape
    assert B == n_bins + 1
    out = np.zeros(n_nodes, dtype=SPLIT_F64_DTYPE)
    st = lib().oracle_find_splits_f64(_ptr(hist), n_nodes, F, n_bins, lam, gamma, min_child_weight, _ptr(out))
    return out, st


def partition(bins: np.ndarray, n_bins: int, sentinel: int, rows, node_offsets, splits: np.ndarray):
    """Route each node's rows into (left 2i, right 2i+1) children; returns (rows, offsets [2n+1], status)."""
    bins = np.ascontiguousarray(bins)
    F, N = bins.shape
    offs = np.ascontiguousarray(node_offsets, dtype=np.int64)
    n_nodes = offs.shape[0] - 1
    rows_a = None if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    total = int(offs[-1] - offs[0]) if n_nodes > 0 else 0
    out_rows = np.empty(total, dtype=np.int32)
    out_offs = np.zeros(2 * n_nodes + 1, dtype=np.int64)
    sp = np.ascontiguousarray(splits, dtype=SPLIT_DTYPE)
    st = lib().oracle_partition(_ptr(bins), bins.dtype.itemsize, N, n_bins, sentinel, _ptr(rows_a), _ptr(offs),
                                n_nodes, _ptr(sp), _ptr(out_rows), _ptr(out_offs))
    return out_rows, out_offs, st
