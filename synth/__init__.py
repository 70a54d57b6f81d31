"""Seeded synthetic inputs for the level histogram path.

This module only draws random inputs and their node structure; it holds none
of the method's arithmetic (no quantisation, histogram, subtraction or gain).
Both the CPU oracle side (tests) and the CUDA side (tests, bench) take their
inputs from here, so the two never feed each other.

Workloads (shapes and distributions follow the pages' benchmark shapes:
"millions of rows, around a hundred features" and the wide 131,072 x 16,384
case of bonsai "E6. The wide-data wall"):

  root      10,000 x 28 u8, bins uniform [0,254], one node holding all rows
  level5    1,000,000 x 100 u8, per-feature Zipf s=1.1 over 255 bins (bin id
            = rank, bin 0 hottest), level 5 of a tree grown by random seeded
            binary partitions (32 nodes, 16 built)
  dense     10,000,000 x 500 u8, uniform bins, h = 0.25, all levels 0..7 of a
            depth-8 tree grown by random seeded partitions
  wide      131,072 x 16,384 u8, uniform bins, level 3 with 8 nodes whose sizes
            are proportional to 0.5 * r^i, r = 0.1^(1/7), over a seeded
            permutation of the rows
  u16miss   2,000,000 x 64 u16, bin = clamp(floor(2048 + 682.7 z), 0, 4095),
            40% of entries set to the sentinel 0xFFFF, level 7 (128 nodes)

Random partition rounds: at every level each node draws p ~ U(0.2, 0.8) and
each of its rows goes left with probability p; children of node i are 2i
(left) and 2i+1 (right). Rows inside a node stay in ascending order.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202

WORKLOADS = {
    "root": dict(cid=1, n_rows=10_000, n_features=28, width=1, n_bins=255, sentinel=0xFF, bins="uniform",
                 h="u0.1", level=0),
    "level5": dict(cid=2, n_rows=1_000_000, n_features=100, width=1, n_bins=255, sentinel=0xFF, bins="zipf",
                   h="u0.05", level=5),
    "dense": dict(cid=3, n_rows=10_000_000, n_features=500, width=1, n_bins=255, sentinel=0xFF, bins="uniform",
                  h="c0.25", level=7),
    "wide": dict(cid=4, n_rows=131_072, n_features=16_384, width=1, n_bins=255, sentinel=0xFF, bins="uniform",
                 h="u0.1", level=3),
    "u16miss": dict(cid=5, n_rows=2_000_000, n_features=64, width=2, n_bins=4096, sentinel=0xFFFF, bins="normal16",
                    h="u0.1", level=7),
}


def rng_for(name: str, salt: int = 0) -> np.random.Generator:
    return np.random.default_rng([SEED_BASE + WORKLOADS[name]["cid"], salt])


# ----------------------------------------------------------------------------- bins
def bins_uniform(rng, n_features, n_rows, n_values=255):
    """Feature-major [F][N] uint8, uniform over [0, n_values).

    For n_values = 255 each feature row is raw random bytes with every 255
    redrawn (rejection sampling: exactly uniform over [0, 254], and fast at GB
    scale)."""
    if n_values != 255:
        return rng.integers(0, n_values, size=(n_features, n_rows), dtype=np.uint8)
    out = np.empty((n_features, n_rows), dtype=np.uint8)
    per = max(1, (64 << 20) // max(n_rows, 1))  # features per 64 MiB block
    for f0 in range(0, n_features, per):
        f1 = min(n_features, f0 + per)
        blk = np.frombuffer(rng.bytes((f1 - f0) * n_rows), dtype=np.uint8).copy()
        bad = np.flatnonzero(blk == 255)
        while bad.size:
            blk[bad] = np.frombuffer(rng.bytes(bad.size), dtype=np.uint8)
            bad = bad[blk[bad] == 255]
        out[f0:f1] = blk.reshape(f1 - f0, n_rows)
    return out


def bins_zipf(rng, n_features, n_rows, s=1.1, n_values=255):
    """Feature-major [F][N] uint8 with P(b) proportional to (b+1)^-s over b in [0, n_values)."""
    w = np.arange(1, n_values + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(w)
    cdf /= cdf[-1]
    out = np.empty((n_features, n_rows), dtype=np.uint8)
    for f in range(n_features):
        u = rng.random(n_rows)
        out[f] = np.minimum(np.searchsorted(cdf, u, side="right"), n_values - 1).astype(np.uint8)
    return out


def bins_normal16(rng, n_features, n_rows, n_bins=4096, missing_frac=0.4, sentinel=0xFFFF):
    """Feature-major [F][N] uint16: clamp(floor(n_bins/2 + n_bins/6 * z)), missing_frac entries -> sentinel."""
    out = np.empty((n_features, n_rows), dtype=np.uint16)
    for f in range(n_features):
        z = rng.standard_normal(n_rows)
        b = np.floor(n_bins / 2 + (n_bins / 6.0) * z)
        b = np.clip(b, 0, n_bins - 1).astype(np.uint16)
        miss = rng.random(n_rows) < missing_frac
        b[miss] = sentinel
        out[f] = b
    return out


def gpair(rng, n_rows, h="u0.1"):
    """Packed float32 (g, h) [N][2]: g ~ N(0,1); h ~ U(lo, 1) for 'u<lo>' or constant for 'c<v>'."""
    out = np.empty((n_rows, 2), dtype=np.float32)
    out[:, 0] = rng.standard_normal(n_rows).astype(np.float32)
    if h.startswith("u"):
        out[:, 1] = rng.uniform(float(h[1:]), 1.0, n_rows).astype(np.float32)
    else:
        out[:, 1] = np.float32(float(h[1:]))
    return out


def fixed_point_scales(gpair_arr, rows_per_partial=65536):
    """The fixed-point scales a workload is run with (an input of the method, chosen from the data):
    for g and h, the largest power of two s with max|x| * s * rows_per_partial <= 2^31 - 1 (1.0 when
    max|x| = 0), clamped to [2^-126, 2^126]."""
    lim = (2 ** 31 - 1) / float(rows_per_partial)
    out = []
    for c in range(2):
        m = float(np.abs(np.asarray(gpair_arr, dtype=np.float32)[..., c]).max()) if np.size(gpair_arr) else 0.0
        if m == 0.0:
            out.append(1.0)
            continue
        e = max(-126, min(126, math.floor(math.log2(lim / m))))
        while e > -126 and m * 2.0 ** e > lim:
            e -= 1
        while e < 126 and m * 2.0 ** (e + 1) <= lim:
            e += 1
        out.append(2.0 ** e)
    return out[0], out[1]


def gpair_multi(name: str, n_rows, k, h="u0.1"):
    """k targets' pairs [N][k][2] float32: target t drawn like `gpair` from its own seeded stream."""
    return np.stack([gpair(rng_for(name, 100 + t), n_rows, h) for t in range(k)], axis=1)


# ----------------------------------------------------------------------------- node structure
def geometric_partition_ids(rng, n_rows, n_nodes=8, lo=0.05, hi=0.5):
    """Node id of every row for n_nodes nodes with sizes proportional to hi * r^i, r = (lo/hi)^(1/(n-1))."""
    r = (lo / hi) ** (1.0 / (n_nodes - 1))
    w = hi * r ** np.arange(n_nodes)
    w = w / w.sum()
    bounds = np.floor(np.cumsum(np.concatenate([[0.0], w])) * n_rows + 0.5).astype(np.int64)
    bounds[-1] = n_rows
    perm = rng.permutation(n_rows)
    node = np.empty(n_rows, dtype=np.int64)
    for i in range(n_nodes):
        node[perm[bounds[i]:bounds[i + 1]]] = i
    return node


def group_rows(node_ids, n_nodes):
    """(rows int32 grouped by node, ascending inside a node; offsets int64 [n_nodes+1])."""
    order = np.argsort(node_ids, kind="stable").astype(np.int32)
    counts = np.bincount(node_ids, minlength=n_nodes)
    offs = np.zeros(n_nodes + 1, dtype=np.int64)
    np.cumsum(counts, out=offs[1:])
    return order, offs


@dataclass
class Level:
    """One tree level: nodes 0..n_nodes-1 with children (2i, 2i+1) of parent i at the level above."""
    depth: int
    rows: np.ndarray          # int32, all rows of the level grouped by node
    offsets: np.ndarray       # int64 [n_nodes + 1]
    # smaller-sibling plan: pair p = nodes (2p, 2p+1), parent p at depth-1
    small: np.ndarray = field(default=None)     # int32 [n_pairs] node id of the built (smaller) sibling
    large: np.ndarray = field(default=None)     # int32 [n_pairs] node id of the derived (larger) sibling
    built_rows: np.ndarray = field(default=None)     # int32 rows of the built nodes, concatenated in pair order
    built_offsets: np.ndarray = field(default=None)  # int64 [n_pairs + 1]

    @property
    def n_nodes(self):
        return self.offsets.shape[0] - 1


def level_from_ids(node_ids, depth, n_nodes):
    rows, offs = group_rows(node_ids, n_nodes)
    lv = Level(depth=depth, rows=rows, offsets=offs)
    if depth > 0:
        sizes = np.diff(offs)
        n_pairs = n_nodes // 2
        left = np.arange(n_pairs) * 2
        right = left + 1
        small = np.where(sizes[right] < sizes[left], right, left).astype(np.int32)  # ties -> left
        large = np.where(small == left, right, left).astype(np.int32)
        parts = [rows[offs[s]:offs[s + 1]] for s in small]
        lv.small, lv.large = small, large
        lv.built_rows = np.concatenate(parts).astype(np.int32) if parts else np.zeros(0, np.int32)
        bo = np.zeros(n_pairs + 1, dtype=np.int64)
        np.cumsum(sizes[small], out=bo[1:])
        lv.built_offsets = bo
    return lv


@dataclass
class Workload:
    name: str
    n_rows: int
    n_features: int
    width: int
    n_bins: int
    sentinel: int
    bins: np.ndarray      # feature-major [F][N]
    gpair: np.ndarray     # float32 [N][2]
    levels: dict          # depth -> Level (the target level and, when it has one, its parent)
    target_depth: int


def make(name: str, n_rows: int | None = None, n_features: int | None = None, depth: int | None = None) -> Workload:
    """Build a workload; n_rows / n_features / depth override the full sizes (reduced parity cases)."""
    spec = dict(WORKLOADS[name])
    N = int(n_rows or spec["n_rows"])
    F = int(n_features or spec["n_features"])
    L = spec["level"] if depth is None else int(depth)
    rng = rng_for(name, 0)
    if spec["bins"] == "uniform":
        bins = bins_uniform(rng, F, N)
    elif spec["bins"] == "zipf":
        bins = bins_zipf(rng, F, N)
    else:
        bins = bins_normal16(rng, F, N, n_bins=spec["n_bins"], sentinel=spec["sentinel"])
    gp = gpair(rng_for(name, 1), N, spec["h"])
    levels = {}
    prng = rng_for(name, 2)
    if name == "wide":
        ids = geometric_partition_ids(prng, N, n_nodes=1 << L)
        levels[L] = level_from_ids(ids, L, 1 << L)
        levels[L - 1] = level_from_ids(ids // 2, L - 1, 1 << (L - 1))
    else:
        node = np.zeros(N, dtype=np.int64)
        levels[0] = level_from_ids(node, 0, 1)
        for d in range(L):
            p = prng.uniform(0.2, 0.8, size=1 << d)
            go_right = prng.random(N) >= p[node]
            node = 2 * node + go_right
            levels[d + 1] = level_from_ids(node, d + 1, 1 << (d + 1))
    return Workload(name=name, n_rows=N, n_features=F, width=spec["width"], n_bins=spec["n_bins"],
                    sentinel=spec["sentinel"], bins=bins, gpair=gp, levels=levels, target_depth=L)
