"""Convenience wrapper over the C ABI for callers that hold data in torch or numpy.

Torch supplies device memory and the stream; every computation is a call into
``libgbthist.so``. Outputs come back as torch tensors (histograms) or numpy
structured arrays (splits).
"""
from __future__ import annotations

import numpy as np

from . import (GBT_OK, SPLIT_BYTES, check, gbt_advance_level, gbt_begin_tree, gbt_begin_tree_multi, gbt_build_level,
               gbt_build_level_f64, gbt_build_level_multi, gbt_create, gbt_partition_level_pairs,
               gbt_destroy, gbt_find_level_split, gbt_find_splits, gbt_find_splits_f64, gbt_kernel_launches,
               gbt_level_step, gbt_partition_level, gbt_subtract_and_find, gbt_subtract_siblings,
               gbt_subtract_siblings_f64, gbt_sync, gbt_upload_bins, lib, params)

SPLIT_DTYPE = np.dtype([
    ("feature", "<i4"), ("bin", "<i4"), ("default_left", "u1"), ("pad", "u1", (7,)), ("gain", "<f8"),
    ("g_left", "<i8"), ("h_left", "<i8"), ("g_right", "<i8"), ("h_right", "<i8"),
])
assert SPLIT_DTYPE.itemsize == SPLIT_BYTES
# float-cell mode: the same record with double sums
SPLIT_F64_DTYPE = np.dtype([
    ("feature", "<i4"), ("bin", "<i4"), ("default_left", "u1"), ("pad", "u1", (7,)), ("gain", "<f8"),
    ("g_left", "<f8"), ("h_left", "<f8"), ("g_right", "<f8"), ("h_right", "<f8"),
])
assert SPLIT_F64_DTYPE.itemsize == SPLIT_BYTES


def splits_to_numpy(t, dtype=SPLIT_DTYPE) -> np.ndarray:
    """A [n, 56] uint8 tensor (device or host) -> numpy structured array of splits."""
    a = t.detach().to("cpu").contiguous().numpy()
    return a.view(dtype).reshape(-1)


class Session:
    """One gbthist context bound to a torch device and stream."""

    def __init__(self, device: int = 0, stream=None):
        import torch
        self.torch = torch
        self.device = torch.device("cuda", device)
        lib()
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        s, h = gbt_create(device, self.stream.cuda_stream)
        check(s)
        self.ctx = h
        self.n_rows = self.n_features = self.n_bins = None

    # -------------------------------------------------------------------- lifetime
    def close(self):
        if self.ctx:
            gbt_destroy(self.ctx)
            self.ctx = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def sync(self) -> int:
        return gbt_sync(self.ctx)

    def check(self, status):
        return check(status, self.ctx)

    @property
    def launches(self) -> int:
        return gbt_kernel_launches(self.ctx)

    # -------------------------------------------------------------------- data
    def upload_bins(self, bins, n_bins: int, sentinel: int):
        """bins: feature-major [F][N] uint8/uint16 numpy array or torch tensor (host or device)."""
        torch = self.torch
        if isinstance(bins, np.ndarray):
            width = bins.dtype.itemsize
            F, N = bins.shape
            arr = np.ascontiguousarray(bins)
            self.check(gbt_upload_bins(self.ctx, arr, width, N, F, n_bins, sentinel))
            self.check(self.sync())  # the host array must stay alive until the copy is done
        else:
            width = bins.element_size()
            F, N = bins.shape
            self.check(gbt_upload_bins(self.ctx, bins.contiguous(), width, N, F, n_bins, sentinel))
        self.n_rows, self.n_features, self.n_bins, self.width = N, F, n_bins, width
        return self

    def begin_tree(self, gpair, scale_g: float, scale_h: float):
        """gpair: [N][2] float32 (numpy host or torch host/device)."""
        if isinstance(gpair, np.ndarray):
            arr = np.ascontiguousarray(gpair, dtype=np.float32)
            self.check(gbt_begin_tree(self.ctx, arr, scale_g, scale_h))
            self.check(self.sync())
        else:
            self.check(gbt_begin_tree(self.ctx, gpair.contiguous(), scale_g, scale_h))
        self.scale_g, self.scale_h = scale_g, scale_h
        return self

    def hist_tensor(self, n_nodes: int):
        return self.torch.empty((n_nodes, self.n_features, self.n_bins + 1, 2), dtype=self.torch.int64,
                                device=self.device)

    def to_dev(self, a, dtype):
        torch = self.torch
        if a is None:
            return None
        if isinstance(a, np.ndarray):
            return torch.from_numpy(np.ascontiguousarray(a)).to(device=self.device, dtype=dtype)
        return a.to(device=self.device, dtype=dtype).contiguous()

    def build_level(self, rows, offsets, hist=None):
        """rows: int32 level list or None (identity); offsets: int64 [n+1]. Returns the int64 histogram tensor."""
        n_nodes = int(len(offsets) - 1)
        if hist is None:
            hist = self.hist_tensor(n_nodes)
        r = self.to_dev(rows, self.torch.int32)
        o = self.to_dev(offsets, self.torch.int64)
        self.check(gbt_build_level(self.ctx, r, o, n_nodes, hist))
        return hist

    def subtract(self, parent, small, parent_of=None, large=None):
        n_pairs = small.shape[0]
        if large is None:
            large = self.torch.empty_like(small)
        po = self.to_dev(parent_of, self.torch.int32)
        self.check(gbt_subtract_siblings(self.ctx, parent, po, small, large, n_pairs))
        return large

    def find_splits(self, hist, lam=1.0, gamma=0.0, mcw=0.0):
        n = hist.shape[0]
        out = self.torch.empty((n, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        self.check(gbt_find_splits(self.ctx, hist, n, params(lam, gamma, mcw), out))
        return out

    def find_level_split(self, hist, lam=1.0, gamma=0.0, mcw=0.0):
        """One oblivious split for all nodes of `hist` ([n][F][B][2] int64): a [1, 56] uint8 tensor."""
        out = self.torch.empty((1, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        self.check(gbt_find_level_split(self.ctx, hist, hist.shape[0], params(lam, gamma, mcw), out))
        return out

    # ------------------------------------------------------- multi-output (vector-leaf) trees
    def begin_tree_multi(self, gpair, scales_g, scales_h):
        """gpair: [N][k][2] float32 (numpy host or torch host/device); one scale pair per target."""
        k = int(len(scales_g))
        if isinstance(gpair, np.ndarray):
            arr = np.ascontiguousarray(gpair, dtype=np.float32)
            self.check(gbt_begin_tree_multi(self.ctx, arr, k, scales_g, scales_h))
            self.check(self.sync())
        else:
            self.check(gbt_begin_tree_multi(self.ctx, gpair.contiguous(), k, scales_g, scales_h))
        self.n_targets = k
        return self

    def build_level_multi(self, rows, offsets, hist=None):
        """Every target's histogram of the level's nodes: [k][n][F][B][2] int64."""
        n_nodes = int(len(offsets) - 1)
        if hist is None:
            hist = self.torch.empty((self.n_targets, n_nodes, self.n_features, self.n_bins + 1, 2),
                                    dtype=self.torch.int64, device=self.device)
        r = self.to_dev(rows, self.torch.int32)
        o = self.to_dev(offsets, self.torch.int64)
        self.check(gbt_build_level_multi(self.ctx, r, o, n_nodes, hist))
        return hist

    # ------------------------------------------------------- float-cell mode
    def build_level_f64(self, gpair, rows, offsets, hist=None):
        """Double-cell histogram of the unquantised float32 gpair ([N][2], host or device): [n][F][B][2] float64."""
        n_nodes = int(len(offsets) - 1)
        if hist is None:
            hist = self.torch.empty((n_nodes, self.n_features, self.n_bins + 1, 2), dtype=self.torch.float64,
                                    device=self.device)
        r = self.to_dev(rows, self.torch.int32)
        o = self.to_dev(offsets, self.torch.int64)
        if isinstance(gpair, np.ndarray):  # host gpair: the library stages it; keep it alive until the copy is done
            gp = np.ascontiguousarray(gpair, dtype=np.float32)
            self.check(gbt_build_level_f64(self.ctx, gp, r, o, n_nodes, hist))
            self.check(self.sync())
        else:
            gp = gpair.to(device=self.device, dtype=self.torch.float32).contiguous()
            self.check(gbt_build_level_f64(self.ctx, gp, r, o, n_nodes, hist))
        return hist

    def subtract_f64(self, parent, small, parent_of=None, large=None):
        n_pairs = small.shape[0]
        if large is None:
            large = self.torch.empty_like(small)
        po = self.to_dev(parent_of, self.torch.int32)
        self.check(gbt_subtract_siblings_f64(self.ctx, parent, po, small, large, n_pairs))
        return large

    def find_splits_f64(self, hist, lam=1.0, gamma=0.0, mcw=0.0):
        n = hist.shape[0]
        out = self.torch.empty((n, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        self.check(gbt_find_splits_f64(self.ctx, hist, n, params(lam, gamma, mcw), out))
        return out

    def subtract_and_find(self, parent, small, parent_of=None, large=None, lam=1.0, gamma=0.0, mcw=0.0):
        n_pairs = small.shape[0]
        if large is None:
            large = self.torch.empty_like(small)
        po = self.to_dev(parent_of, self.torch.int32)
        so = self.torch.empty((n_pairs, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        lo = self.torch.empty((n_pairs, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        self.check(gbt_subtract_and_find(self.ctx, parent, po, small, large, n_pairs, params(lam, gamma, mcw), so, lo))
        return large, so, lo

    def level_step(self, rows, offsets, parent, parent_of=None, small=None, large=None, lam=1.0, gamma=0.0, mcw=0.0):
        """Build the smaller siblings (rows/offsets: one segment per pair), subtract, find splits of both."""
        n_pairs = int(len(offsets) - 1)
        if small is None:
            small = self.hist_tensor(n_pairs)
        if large is None:
            large = self.torch.empty_like(small)
        r = self.to_dev(rows, self.torch.int32)
        o = self.to_dev(offsets, self.torch.int64)
        po = self.to_dev(parent_of, self.torch.int32)
        so = self.torch.empty((n_pairs, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        lo = self.torch.empty((n_pairs, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        self.check(gbt_level_step(self.ctx, r, o, n_pairs, parent, po, small, large, params(lam, gamma, mcw), so, lo))
        return small, large, so, lo

    def partition(self, rows, offsets, splits):
        """splits: [n, 56] uint8 tensor or numpy SPLIT_DTYPE array. Returns (rows, offsets [2n+1]) tensors."""
        torch = self.torch
        n_nodes = int(len(offsets) - 1)
        R = int(offsets[-1])
        r = self.to_dev(rows, torch.int32)
        o = self.to_dev(offsets, torch.int64)
        if isinstance(splits, np.ndarray):
            splits = torch.from_numpy(np.ascontiguousarray(splits).view(np.uint8).reshape(-1, SPLIT_BYTES)).to(
                self.device)
        out_rows = torch.empty(max(R, 1), dtype=torch.int32, device=self.device)
        out_offs = torch.empty(2 * n_nodes + 1, dtype=torch.int64, device=self.device)
        self.check(gbt_partition_level(self.ctx, r, o, n_nodes, splits, out_rows, out_offs))
        return out_rows[:R], out_offs

    def partition_pairs(self, rows, offsets, splits, n_rows_level=None):
        """gbt_partition_level_pairs: returns (rows, offsets [2n+1], small_rows, small_offsets [n+1],
        small_side [n]) device tensors. n_rows_level: the level's row count (read from offsets if None)."""
        torch = self.torch
        n_nodes = int(len(offsets) - 1)
        R = int(offsets[-1]) if n_rows_level is None else int(n_rows_level)
        r = self.to_dev(rows, torch.int32)
        o = self.to_dev(offsets, torch.int64)
        if isinstance(splits, np.ndarray):
            splits = torch.from_numpy(np.ascontiguousarray(splits).view(np.uint8).reshape(-1, SPLIT_BYTES)).to(
                self.device)
        out_rows = torch.empty(max(R, 1), dtype=torch.int32, device=self.device)
        out_offs = torch.empty(2 * n_nodes + 1, dtype=torch.int64, device=self.device)
        small_rows = torch.empty(max(R // 2, 1), dtype=torch.int32, device=self.device)
        small_offs = torch.empty(n_nodes + 1, dtype=torch.int64, device=self.device)
        small_side = torch.empty(n_nodes, dtype=torch.uint8, device=self.device)
        self.check(gbt_partition_level_pairs(self.ctx, r, o, n_nodes, splits, out_rows, out_offs, small_rows,
                                             small_offs, small_side))
        return out_rows[:R], out_offs, small_rows, small_offs, small_side

    def advance_level(self, small_rows, small_offsets, small_side, parent, level_hist=None, lam=1.0, gamma=0.0,
                      mcw=0.0, splits=None):
        """gbt_advance_level: the next level's histograms and splits in node order ([2 n_pairs] each)."""
        n_pairs = parent.shape[0]
        if level_hist is None:
            level_hist = self.hist_tensor(2 * n_pairs)
        if splits is None:
            splits = self.torch.empty((2 * n_pairs, SPLIT_BYTES), dtype=self.torch.uint8, device=self.device)
        self.check(gbt_advance_level(self.ctx, small_rows, small_offsets, small_side, n_pairs, parent, level_hist,
                                     params(lam, gamma, mcw), splits))
        return level_hist, splits
