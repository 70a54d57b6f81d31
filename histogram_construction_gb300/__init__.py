"""Python binding of the gbthist C ABI (``include/gbthist.h``).

Argument marshalling only: every step of the histogram path runs in the CUDA
kernels of ``libgbthist.so``. Pointers may be torch tensors (device or host),
numpy arrays (host), ``None`` or raw integer addresses. Functions return the
``gbt_status`` code; :func:`check` turns a non-zero code into an exception.
There is no fallback: if the library is missing, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

GBT_OK = 0
STATUS_NAMES = {
    0: "GBT_OK", 1: "GBT_ERR_INVALID_ARG", 2: "GBT_ERR_STATE", 3: "GBT_ERR_OOM", 4: "GBT_ERR_CUDA",
    5: "GBT_ERR_BIN_RANGE", 6: "GBT_ERR_ROW_RANGE", 7: "GBT_ERR_QUANT_OVERFLOW", 8: "GBT_ERR_UNSUPPORTED",
    9: "GBT_ERR_TIMEOUT", 10: "GBT_ERR_INCONSISTENT",
}
(GBT_ERR_INVALID_ARG, GBT_ERR_STATE, GBT_ERR_OOM, GBT_ERR_CUDA, GBT_ERR_BIN_RANGE, GBT_ERR_ROW_RANGE,
 GBT_ERR_QUANT_OVERFLOW, GBT_ERR_UNSUPPORTED, GBT_ERR_TIMEOUT, GBT_ERR_INCONSISTENT) = range(1, 11)

EXPORTS = [
    "gbt_create", "gbt_destroy", "gbt_last_error", "gbt_sync", "gbt_upload_bins", "gbt_begin_tree",
    "gbt_suggest_scales", "gbt_build_level", "gbt_subtract_siblings", "gbt_find_splits", "gbt_subtract_and_find",
    "gbt_level_step",
    "gbt_partition_level", "gbt_profile_enable", "gbt_profile_read", "gbt_slots_per_feature",
    "gbt_kernel_launches", "gbt_find_splits_noalloc", "gbt_find_level_split", "gbt_build_level_f64",
    "gbt_subtract_siblings_f64", "gbt_find_splits_f64", "gbt_begin_tree_multi", "gbt_build_level_multi",
    "gbt_partition_level_pairs", "gbt_advance_level",
]


class GbtSplit(ctypes.Structure):
    _fields_ = [
        ("feature", ctypes.c_int32), ("bin", ctypes.c_int32), ("default_left", ctypes.c_uint8),
        ("pad", ctypes.c_uint8 * 7), ("gain", ctypes.c_double), ("g_left", ctypes.c_int64),
        ("h_left", ctypes.c_int64), ("g_right", ctypes.c_int64), ("h_right", ctypes.c_int64),
    ]


class GbtParams(ctypes.Structure):
    _fields_ = [("lambda_", ctypes.c_double), ("gamma", ctypes.c_double), ("min_child_weight", ctypes.c_double)]


SPLIT_BYTES = ctypes.sizeof(GbtSplit)
assert SPLIT_BYTES == 56

_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def lib(build_if_missing: bool = True):
    """Load libgbthist.so (building it first if needed). Raises if it cannot be had."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"gbthist library not built: {path}")
    L = ctypes.CDLL(path)
    vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    st = ctypes.c_int
    sig = {
        "gbt_create": (st, [ctypes.c_int, vp, ctypes.POINTER(vp)]),
        "gbt_destroy": (st, [vp]),
        "gbt_last_error": (ctypes.c_char_p, [vp]),
        "gbt_sync": (st, [vp]),
        "gbt_upload_bins": (st, [vp, vp, ctypes.c_int, i64, i32, i32, ctypes.c_uint32]),
        "gbt_begin_tree": (st, [vp, vp, f32, f32]),
        "gbt_suggest_scales": (st, [i64, f32, f32, ctypes.POINTER(f32), ctypes.POINTER(f32)]),
        "gbt_build_level": (st, [vp, vp, vp, i32, vp]),
        "gbt_subtract_siblings": (st, [vp, vp, vp, vp, vp, i32]),
        "gbt_find_splits": (st, [vp, vp, i32, ctypes.POINTER(GbtParams), vp]),
        "gbt_subtract_and_find": (st, [vp, vp, vp, vp, vp, i32, ctypes.POINTER(GbtParams), vp, vp]),
        "gbt_level_step": (st, [vp, vp, vp, i32, vp, vp, vp, vp, ctypes.POINTER(GbtParams), vp, vp]),
        "gbt_partition_level": (st, [vp, vp, vp, i32, vp, vp, vp]),
        "gbt_partition_level_pairs": (st, [vp, vp, vp, i32, vp, vp, vp, vp, vp, vp]),
        "gbt_advance_level": (st, [vp, vp, vp, vp, i32, vp, vp, ctypes.POINTER(GbtParams), vp]),
        "gbt_profile_enable": (st, [vp, ctypes.c_int]),
        "gbt_profile_read": (st, [vp, ctypes.c_char_p, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i64)]),
        "gbt_slots_per_feature": (i32, [vp]),
        "gbt_kernel_launches": (i64, [vp]),
        "gbt_find_splits_noalloc": (st, [vp, i32, i32, i32, f32, f32, ctypes.POINTER(GbtParams), vp, vp]),
        "gbt_find_level_split": (st, [vp, vp, i32, ctypes.POINTER(GbtParams), vp]),
        "gbt_build_level_f64": (st, [vp, vp, vp, vp, i32, vp]),
        "gbt_begin_tree_multi": (st, [vp, vp, i32, vp, vp]),
        "gbt_build_level_multi": (st, [vp, vp, vp, i32, vp]),
        "gbt_subtract_siblings_f64": (st, [vp, vp, vp, vp, vp, i32]),
        "gbt_find_splits_f64": (st, [vp, vp, i32, ctypes.POINTER(GbtParams), vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return _lib


def ptr(x):
    """Address of a torch tensor / numpy array / ctypes object / int, or None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    return ctypes.addressof(x)


class GbtError(RuntimeError):
    def __init__(self, status, msg=""):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def check(status, ctx=None):
    if status != GBT_OK:
        msg = ""
        if ctx is not None:
            m = lib().gbt_last_error(ctx)
            msg = m.decode() if m else ""
        raise GbtError(status, msg)
    return status


def params(lam=1.0, gamma=0.0, min_child_weight=0.0) -> GbtParams:
    return GbtParams(float(lam), float(gamma), float(min_child_weight))


# ----------------------------------------------------------------------------- same-name wrappers
def gbt_create(device=0, stream=None):
    h = ctypes.c_void_p()
    s = lib().gbt_create(int(device), ptr(stream), ctypes.byref(h))
    return s, h.value


def gbt_destroy(ctx):
    return lib().gbt_destroy(ctx)


def gbt_last_error(ctx) -> str:
    m = lib().gbt_last_error(ctx)
    return m.decode() if m else ""


def gbt_sync(ctx):
    return lib().gbt_sync(ctx)


def gbt_upload_bins(ctx, bins, bin_bytes, n_rows, n_features, n_bins, missing_sentinel):
    return lib().gbt_upload_bins(ctx, ptr(bins), int(bin_bytes), int(n_rows), int(n_features), int(n_bins),
                                 int(missing_sentinel))


def gbt_begin_tree(ctx, gpair, scale_g, scale_h):
    return lib().gbt_begin_tree(ctx, ptr(gpair), float(scale_g), float(scale_h))


def gbt_suggest_scales(rows_per_partial, max_abs_g, max_abs_h):
    sg, sh = ctypes.c_float(), ctypes.c_float()
    s = lib().gbt_suggest_scales(int(rows_per_partial), float(max_abs_g), float(max_abs_h), ctypes.byref(sg),
                                 ctypes.byref(sh))
    return s, sg.value, sh.value


def gbt_build_level(ctx, rows, node_offsets, n_nodes, hist_out):
    return lib().gbt_build_level(ctx, ptr(rows), ptr(node_offsets), int(n_nodes), ptr(hist_out))


def gbt_subtract_siblings(ctx, parent_hist, parent_of, small_hist, large_hist, n_pairs):
    return lib().gbt_subtract_siblings(ctx, ptr(parent_hist), ptr(parent_of), ptr(small_hist), ptr(large_hist),
                                       int(n_pairs))


def gbt_find_splits(ctx, hist, n_nodes, prm, out):
    return lib().gbt_find_splits(ctx, ptr(hist), int(n_nodes), ctypes.byref(prm), ptr(out))


def gbt_begin_tree_multi(ctx, gpair, n_targets, scales_g, scales_h):
    sg = (ctypes.c_float * int(n_targets))(*[float(x) for x in scales_g])
    sh = (ctypes.c_float * int(n_targets))(*[float(x) for x in scales_h])
    return lib().gbt_begin_tree_multi(ctx, ptr(gpair), int(n_targets), ctypes.cast(sg, ctypes.c_void_p),
                                      ctypes.cast(sh, ctypes.c_void_p))


def gbt_build_level_multi(ctx, rows, node_offsets, n_nodes, hist_out):
    return lib().gbt_build_level_multi(ctx, ptr(rows), ptr(node_offsets), int(n_nodes), ptr(hist_out))


def gbt_build_level_f64(ctx, gpair, rows, node_offsets, n_nodes, hist_out):
    return lib().gbt_build_level_f64(ctx, ptr(gpair), ptr(rows), ptr(node_offsets), int(n_nodes), ptr(hist_out))


def gbt_subtract_siblings_f64(ctx, parent_hist, parent_of, small_hist, large_hist, n_pairs):
    return lib().gbt_subtract_siblings_f64(ctx, ptr(parent_hist), ptr(parent_of), ptr(small_hist), ptr(large_hist),
                                           int(n_pairs))


def gbt_find_splits_f64(ctx, hist, n_nodes, prm, out):
    return lib().gbt_find_splits_f64(ctx, ptr(hist), int(n_nodes), ctypes.byref(prm), ptr(out))


def gbt_find_level_split(ctx, hist, n_nodes, prm, out):
    return lib().gbt_find_level_split(ctx, ptr(hist), int(n_nodes), ctypes.byref(prm), ptr(out))


def gbt_find_splits_noalloc(hist, n_nodes, n_features, n_bins, scale_g, scale_h, prm, out, stream=None):
    """Context-free split find that allocates nothing (device hist and out; see the header for its limits)."""
    return lib().gbt_find_splits_noalloc(ptr(hist), int(n_nodes), int(n_features), int(n_bins), float(scale_g),
                                         float(scale_h), ctypes.byref(prm), ptr(out), stream)


def gbt_subtract_and_find(ctx, parent_hist, parent_of, small_hist, large_hist, n_pairs, prm, small_out, large_out):
    return lib().gbt_subtract_and_find(ctx, ptr(parent_hist), ptr(parent_of), ptr(small_hist), ptr(large_hist),
                                       int(n_pairs), ctypes.byref(prm), ptr(small_out), ptr(large_out))


def gbt_level_step(ctx, rows, node_offsets, n_pairs, parent_hist, parent_of, small_hist, large_hist, prm, small_out,
                   large_out):
    return lib().gbt_level_step(ctx, ptr(rows), ptr(node_offsets), int(n_pairs), ptr(parent_hist), ptr(parent_of),
                                ptr(small_hist), ptr(large_hist), ctypes.byref(prm), ptr(small_out), ptr(large_out))


def gbt_partition_level(ctx, rows, node_offsets, n_nodes, splits, out_rows, out_offsets):
    return lib().gbt_partition_level(ctx, ptr(rows), ptr(node_offsets), int(n_nodes), ptr(splits), ptr(out_rows),
                                     ptr(out_offsets))


def gbt_partition_level_pairs(ctx, rows, node_offsets, n_nodes, splits, out_rows, out_offsets, small_rows,
                              small_offsets, small_side):
    return lib().gbt_partition_level_pairs(ctx, ptr(rows), ptr(node_offsets), int(n_nodes), ptr(splits),
                                           ptr(out_rows), ptr(out_offsets), ptr(small_rows), ptr(small_offsets),
                                           ptr(small_side))


def gbt_advance_level(ctx, small_rows, small_offsets, small_side, n_pairs, parent_hist, level_hist, prm,
                      level_splits):
    return lib().gbt_advance_level(ctx, ptr(small_rows), ptr(small_offsets), ptr(small_side), int(n_pairs),
                                   ptr(parent_hist), ptr(level_hist), ctypes.byref(prm), ptr(level_splits))


def gbt_profile_enable(ctx, on=True):
    return lib().gbt_profile_enable(ctx, 1 if on else 0)


def gbt_profile_read(ctx, kernel=None):
    """Returns (status, total_ms, launches) for `kernel` (name) or all kernels since the last read."""
    ms, n = ctypes.c_double(), ctypes.c_int64()
    s = lib().gbt_profile_read(ctx, kernel.encode() if kernel else None, ctypes.byref(ms), ctypes.byref(n))
    return s, ms.value, n.value


def gbt_slots_per_feature(ctx):
    return lib().gbt_slots_per_feature(ctx)


def gbt_kernel_launches(ctx):
    return lib().gbt_kernel_launches(ctx)
