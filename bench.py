#!/usr/bin/env python
"""Benchmark of the level histogram path: binned entries per second per level on GB300.

One step = one tree level of the workload through gbt_level_step: the
histograms of the smaller siblings (level plan + histogram kernel), sibling
subtraction and split find for both siblings of every pair (level-finish
kernel). ``--path unfused`` times gbt_build_level + gbt_subtract_and_find
instead. Inputs are resident in HBM when the timed region starts; L2 is
flushed (a write larger than L2) before every step, outside the step's CUDA
events.

Prints one JSON line (rank 0): the headline workload (level5 by default) and,
unless ``--no-per-config``, a ``per_config`` object with the other workloads:
root, wide, u16miss and the dense depth-8 tree grown level by level on the
device. ``--impl reference`` times the serial CPU oracle on the headline
workload instead (rank 0 only).

Algorithmic bytes (the roofline's numerator), with R rows in built nodes, F
features, w bytes per bin, B slots per feature, n_b built nodes and n_p
sibling pairs:
  histogram kernel  R*F*w + R*12 (row id, qg, qh) + n_b*F*B*16 (int64 cells)
  level step        the above + 3*n_p*F*B*16 (read parent, read small, write large)
  root level        N*F*w + N*8 + F*B*16 (kernel), + F*B*16 more (split find reads it)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "binned entries/sec per level histogram build (1 GB300); % of HBM roofline"
UNIT = "entries/s"
WORKLOAD_TEXT = {
    "level5": "level5: 1,000,000 rows x 100 features u8 (per-feature Zipf s=1.1 over 255 bins), level 5 of a tree "
              "grown by random seeded partitions: 16 smaller siblings built, 16 derived by subtraction, split find "
              "for all 32",
    "wide": "wide: 131,072 rows x 16,384 features u8 uniform, level 3 with 8 nodes of geometric sizes: 4 built, "
            "4 derived, split find for all 8",
    "u16miss": "u16miss: 2,000,000 rows x 64 features u16 (4096 bins, 40% missing), level 7: 64 built, 64 derived, "
               "split find for all 128",
    "root": "root: 10,000 rows x 28 features u8 uniform, one node (identity rows), build + split find",
    "dense": "dense: 10,000,000 rows x 500 features u8 uniform, h = 0.25, a depth-8 tree (levels 0-7) grown on the "
             "device by its own splits: root build + split find, then per level the row partition and the level "
             "step (smaller siblings built, larger derived, split find for all)",
}
PER_CONFIG = ("root", "wide", "u16miss", "dense")


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _kernel_source_hash():
    h = hashlib.sha256()
    for name in ("k_hist.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "histogram_construction_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profile_traffic(workload):
    """DRAM bytes per launch of the histogram kernel from a committed ncu summary, if it matches the source."""
    path = os.path.join(ROOT, "profiles", f"k_hist_u8_{workload}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("source_hash") == _kernel_source_hash():
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.12)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), smax=float(parts[2]), hw=parts[5], hwt=parts[6], swt=parts[7],
                                 pcap=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for k, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                            ("pcap", "sw_power_cap")):
                if r[k].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["smax"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# ----------------------------------------------------------------------------- workload setup
def level_plan(w: synth.Workload):
    """(parent level, target level) row lists for the bench level of a workload."""
    L = w.target_depth
    if L == 0:
        return None, w.levels[0]
    return w.levels[L - 1], w.levels[L]


def algorithmic_bytes(R, F, wb, B, n_b, n_p, root=False):
    """(histogram kernel bytes, level step bytes) per launch / step (formulas in the module docstring)."""
    if root:
        kernel = R * F * wb + R * 8 + n_b * F * B * 16
        return kernel, kernel + n_b * F * B * 16
    kernel = R * F * wb + R * 12 + n_b * F * B * 16
    return kernel, kernel + 3 * n_p * F * B * 16


def entries_and_bytes(w, lv, B):
    """Units of one step and its algorithmic HBM bytes (histogram kernel, whole level)."""
    F, wb = w.n_features, w.width
    if lv.depth == 0:
        R = int(lv.offsets[-1])
        n_b, n_p = 1, 0
    else:
        R = int(lv.built_offsets[-1])
        n_b = n_p = len(lv.small)
    kernel_bytes, level_bytes = algorithmic_bytes(R, F, wb, B, n_b, n_p, root=lv.depth == 0)
    return R * F, R, n_b, n_p, kernel_bytes, level_bytes


def scales_for(w):
    """The workload's fixed-point scales (equal to gbt_suggest_scales on the same data; tests/test_abi.py)."""
    return synth.fixed_point_scales(w.gpair)


# ----------------------------------------------------------------------------- CPU legs
def oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice=None):
    """Serial oracle for one step: build the smaller siblings, subtract, find splits for both.
    node_slice restricts the step to a prefix of the built nodes (bounded sample)."""
    if lv.depth == 0:
        h, _ = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, None, lv.offsets)
        oracle.find_splits(h, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
        return int(lv.offsets[-1]) * w.n_features
    k = len(lv.small) if node_slice is None else node_slice
    offs = lv.built_offsets[:k + 1]
    rows = lv.built_rows[:int(offs[-1])]
    hs, _ = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, rows, offs)
    large, _ = oracle.subtract(parent_hist[:k], None, hs)
    oracle.find_splits(hs, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
    oracle.find_splits(large, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
    return int(offs[-1]) * w.n_features


def cpu_oracle_timing(w, budget_s=10.0, steps=None, warmup=0, lv=None, parent_rows=None):
    """Time the oracle as it stands (1 thread). Returns (entries/s, sample text, per-step seconds).
    lv / parent_rows override the workload's bench level (a level and its parents' (rows, offsets))."""
    import oracle
    sg, sh = scales_for(w)
    q, _ = oracle.quantise(w.gpair, sg, sh)
    if lv is None:
        par, lv = level_plan(w)
        parent_rows = None if par is None else (par.rows, par.offsets)
    parent_hist = None
    if parent_rows is not None:
        parent_hist, _ = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, parent_rows[0], parent_rows[1])
    n_nodes = len(lv.small) if lv.depth > 0 else 1
    # calibrate on one built node (or the root), then size the sample to the budget
    t0 = time.perf_counter()
    e1 = oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice=1 if lv.depth > 0 else None)
    t1 = time.perf_counter() - t0
    n_total = (steps + warmup) if steps is not None else 1
    node_slice = None
    if lv.depth > 0:
        per_node = t1
        k = int(budget_s / max(per_node * n_total, 1e-9))
        node_slice = None if k >= n_nodes else max(1, k)
    what = "the full level" if node_slice is None else f"the first {node_slice} of {n_nodes} built nodes"
    if steps is not None:
        for _ in range(warmup):
            oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice)
        ent, per = 0, []
        t0 = time.perf_counter()
        for _ in range(steps):
            ts = time.perf_counter()
            ent += oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice)
            per.append(time.perf_counter() - ts)
        dt = time.perf_counter() - t0
        return ent / dt, f"{steps} steps of {what} ({ent // steps} entries per step: build, subtract, split find)", per
    reps, ent, dt = 0, 0, 0.0
    while dt < budget_s or reps == 0:
        t0 = time.perf_counter()
        ent += oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice)
        dt += time.perf_counter() - t0
        reps += 1
        if dt > 0.5 * budget_s and reps >= 1 and node_slice is not None:
            break
    return ent / dt, f"{what} ({ent // reps} entries: build, subtract, split find) x {reps} repetitions", None


def cpu_openmp_timing(w, budget_s=5.0, lv=None, parent_rows=None):
    """The all-core OpenMP baseline (feature-parallel fill, subtraction, serial split scan) on a bounded
    sample of the same level. Returns a cpu_baseline-style dict, or one with 'unavailable'."""
    try:
        import cpu_baseline
        threads = cpu_baseline.threads()
    except Exception as e:  # no OpenMP toolchain on this host
        return {"kind": "openmp", "unavailable": f"{type(e).__name__}: {e}"[:200]}
    sg, sh = scales_for(w)
    q = cpu_baseline.quantise(w.gpair, sg, sh)
    if lv is None:
        par, lv = level_plan(w)
        parent_rows = None if par is None else (par.rows, par.offsets)
    parent = None
    if parent_rows is not None:
        parent, _, _, _ = cpu_baseline.level(w.bins, w.n_bins, w.sentinel, q, parent_rows[0], parent_rows[1])
    if lv.depth == 0:
        rows, offs, n_nodes = None, lv.offsets, 1
    else:
        rows, offs, n_nodes = lv.built_rows, lv.built_offsets, len(lv.small)

    def run(k):
        o = offs[:k + 1]
        r = None if rows is None else rows[:int(o[-1])]
        p = None if parent is None else parent[:k]
        cpu_baseline.level(w.bins, w.n_bins, w.sentinel, q, r, o, p, 1.0, 0.0, 0.0, sg, sh)
        return int(o[-1]) * w.n_features

    t0 = time.perf_counter()
    run(1)
    t1 = time.perf_counter() - t0
    k = n_nodes if n_nodes == 1 else max(1, min(n_nodes, int(budget_s / 3 / max(t1, 1e-9))))
    reps, ent, dt = 0, 0, 0.0
    while dt < budget_s * 0.5 or reps < 2:
        t0 = time.perf_counter()
        ent += run(k)
        dt += time.perf_counter() - t0
        reps += 1
        if dt > budget_s:
            break
    what = "the full level" if k == n_nodes else f"the first {k} of {n_nodes} built nodes"
    return {"value": ent / dt, "unit": UNIT, "cores": threads, "kind": "openmp",
            "sample": f"{what} ({ent // reps} entries: fill, subtract, serial split scan) x {reps} repetitions",
            "nproc": os.cpu_count()}


# ----------------------------------------------------------------------------- GPU leg
def aggregate_ranks(total_ms, e2e_value, world, dist=None, device=None):
    """Whole-job timing over replicas: the slowest rank's timed total (MAX) and the
    slowest rank's end-to-end rate (MIN per rank, times world). Every rank calls it."""
    if dist is None or world == 1:
        return total_ms, e2e_value
    import torch
    t = torch.tensor([total_ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    e = torch.tensor([e2e_value / world], device=device, dtype=torch.float64)
    dist.all_reduce(e, op=dist.ReduceOp.MIN)
    return float(t.item()), float(e.item()) * world


def job_throughput(world, steps, entries_per_rank_step, total_ms):
    """Units all ranks processed divided by the slowest rank's time (weak scaling)."""
    return world * steps * entries_per_rank_step / (total_ms / 1e3)


class Timer:
    """CUDA-event timing of a step callable on one stream, L2 flushed before every step (outside the events)."""

    def __init__(self, torch, stream, dev, g, ctx):
        self.torch, self.stream, self.g, self.ctx = torch, stream, g, ctx
        prop = torch.cuda.get_device_properties(dev)
        self.l2 = int(getattr(prop, "L2_cache_size", 0) or 0) or (129 << 20)
        self.flush_buf = torch.empty(2 * self.l2, dtype=torch.uint8, device=dev)

    def flush(self, i):
        self.flush_buf.fill_(i & 0xFF)

    def run(self, step, steps, warmup=3, flush_l2=True, profile_kernels=None):
        """Returns (per-step ms list, launches of this library in the timed steps, {kernel: ms per launch})."""
        torch, g, ctx = self.torch, self.g, self.ctx
        for i in range(warmup):
            self.flush(i)
            step()
        torch.cuda.synchronize()
        if profile_kernels:
            g.gbt_profile_enable(ctx, True)
            g.gbt_profile_read(ctx)  # forget earlier records
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        l0 = g.gbt_kernel_launches(ctx)
        for i in range(steps):
            if flush_l2:
                self.flush(i)
            ev[i][0].record(self.stream)
            step()
            ev[i][1].record(self.stream)
        torch.cuda.synchronize()
        launches = g.gbt_kernel_launches(ctx) - l0
        kern = {}
        if profile_kernels:
            for name in profile_kernels:
                _, t, n = g.gbt_profile_read(ctx, name)
                if n:
                    kern[name] = t / n
            g.gbt_profile_enable(ctx, False)
        return [a.elapsed_time(b) for a, b in ev], launches, kern


def roofline_obj(kernel, kernel_bytes, kernel_ms, peak, peak_kind, traffic=None):
    achieved = kernel_bytes / (kernel_ms / 1e3) / 1e9 if kernel_ms else None
    return {"bound": "hbm", "kernel": kernel, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": (achieved / peak) if achieved else None, "traffic": traffic,
            "algorithmic_bytes_per_launch": kernel_bytes, "avg_launch_ms": kernel_ms,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"}


def level_summary(ms, entries, level_bytes, peak):
    t = statistics.mean(ms)
    return {"ms_per_step": t, "median_ms_per_step": statistics.median(ms), "entries_per_step": entries,
            "value": entries / (t / 1e3), "unit": UNIT,
            "level_roofline": {"algorithmic_bytes_per_step": level_bytes,
                               "achieved_gbs": level_bytes / (t / 1e3) / 1e9,
                               "frac": level_bytes / (t / 1e3) / 1e9 / peak, "peak": peak}}


KERNELS = ["k_gather_q", "k_hist_u8", "k_hist_u16", "k_level_plan", "k_subtract_find", "k_level_finish", "k_finalize", "k_find",
           "k_part_flags", "k_part_scan", "k_part_scatter"]


def run_config_level(name, torch, g, dev, stream, args, peak, peak_kind):
    """One workload's bench level (the headline's shape) on a fresh context: timing, roofline, CPU baselines."""
    from histogram_construction_gb300.session import Session
    w = synth.make(name)
    sg, sh = scales_for(w)
    par, lv = level_plan(w)
    B = w.n_bins + 1
    entries, R, n_b, n_p, kernel_bytes, level_bytes = entries_and_bytes(w, lv, B)
    hist_kernel = "k_hist_u8" if w.width == 1 else "k_hist_u16"
    out = {"workload": WORKLOAD_TEXT[name]}
    with torch.cuda.stream(stream):
        sess = Session(dev.index, stream=stream)
        sess.upload_bins(torch.from_numpy(w.bins).to(dev), w.n_bins, w.sentinel)
        sess.begin_tree(torch.from_numpy(w.gpair).to(dev), sg, sh)
        prm = g.params(1.0, 0.0, 0.0)
        ctx = sess.ctx
        if lv.depth > 0:
            hp = sess.build_level(torch.from_numpy(par.rows).to(dev), torch.from_numpy(par.offsets).to(dev))
            rows_d = torch.from_numpy(lv.built_rows).to(dev)
            offs_d = torch.from_numpy(lv.built_offsets).to(dev)
            hs, large = sess.hist_tensor(n_b), sess.hist_tensor(n_b)
            so = torch.empty((n_p, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)
            lo = torch.empty_like(so)

            def step():
                sess.check(g.gbt_level_step(ctx, rows_d, offs_d, n_p, hp, None, hs, large, prm, so, lo))
        else:
            offs_d = torch.from_numpy(lv.offsets).to(dev)
            hs = sess.hist_tensor(1)
            so = torch.empty((1, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)

            def step():
                sess.check(g.gbt_build_level(ctx, None, offs_d, 1, hs))
                sess.check(g.gbt_find_splits(ctx, hs, 1, prm, so))
        tm = Timer(torch, stream, dev, g, ctx)
        ms, launches, _ = tm.run(step, args.cfg_steps, warmup=args.warmup)
        _, _, kern = tm.run(step, args.cfg_steps, warmup=1, profile_kernels=KERNELS)
        assert sess.sync() == 0
        sess.close()
        del tm
    out.update(level_summary(ms, entries, level_bytes, peak))
    out["gpu_launches_per_step"] = launches / len(ms)
    out["kernels_ms_per_launch"] = kern
    out["roofline"] = roofline_obj(hist_kernel, kernel_bytes, kern.get(hist_kernel), peak, peak_kind)
    cv, csample, _ = cpu_oracle_timing(w, budget_s=args.cpu_budget)
    out["cpu_baseline"] = {"value": cv, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": csample}
    out["cpu_baseline_openmp"] = cpu_openmp_timing(w, budget_s=args.cpu_budget)
    torch.cuda.empty_cache()
    return out


def run_dense_tree(torch, g, dev, stream, args, peak, peak_kind):
    """The dense workload's depth-8 tree grown on the device by its own splits; each level timed on its own
    (the level step, and the partition that feeds it), and the whole tree."""
    from histogram_construction_gb300.session import Session
    name = "dense"
    w = synth.make(name, depth=0)
    sg, sh = scales_for(w)
    N, F, B, wb = w.n_rows, w.n_features, w.n_bins + 1, w.width
    depth = 7
    out = {"workload": WORKLOAD_TEXT[name], "levels": []}
    with torch.cuda.stream(stream):
        sess = Session(dev.index, stream=stream)
        bins_d = torch.from_numpy(w.bins).to(dev)
        sess.upload_bins(bins_d, w.n_bins, w.sentinel)
        sess.begin_tree(torch.from_numpy(w.gpair).to(dev), sg, sh)
        torch.cuda.synchronize()
        del bins_d
        prm = g.params(1.0, 0.0, 0.0)
        ctx = sess.ctx
        offs0 = torch.tensor([0, N], dtype=torch.int64, device=dev)
        # grow once, keeping every level's buffers (device only)
        lvl = [{"offs": offs0, "rows": None, "hist": sess.hist_tensor(1),
                "splits": torch.empty((1, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)}]

        def root_step():
            sess.check(g.gbt_build_level(ctx, None, offs0, 1, lvl[0]["hist"]))
            sess.check(g.gbt_find_splits(ctx, lvl[0]["hist"], 1, prm, lvl[0]["splits"]))

        root_step()
        for d in range(1, depth + 1):
            n_par = 1 << (d - 1)
            L = {"rows": torch.empty(N, dtype=torch.int32, device=dev),
                 "offs": torch.empty(2 * n_par + 1, dtype=torch.int64, device=dev),
                 "srows": torch.empty(N // 2 + 1, dtype=torch.int32, device=dev),
                 "soffs": torch.empty(n_par + 1, dtype=torch.int64, device=dev),
                 "sside": torch.empty(n_par, dtype=torch.uint8, device=dev),
                 "hist": sess.hist_tensor(2 * n_par),
                 "splits": torch.empty((2 * n_par, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)}
            lvl.append(L)

        def part_step(d):
            P, L = lvl[d - 1], lvl[d]
            sess.check(g.gbt_partition_level_pairs(ctx, P["rows"], P["offs"], 1 << (d - 1), P["splits"], L["rows"],
                                                   L["offs"], L["srows"], L["soffs"], L["sside"]))

        def adv_step(d):
            P, L = lvl[d - 1], lvl[d]
            sess.check(g.gbt_advance_level(ctx, L["srows"], L["soffs"], L["sside"], 1 << (d - 1), P["hist"],
                                           L["hist"], prm, L["splits"]))

        def tree_step():
            root_step()
            for d in range(1, depth + 1):
                part_step(d)
                adv_step(d)

        tree_step()
        assert sess.sync() == 0
        built = [N] + [int(lvl[d]["soffs"][-1].item()) for d in range(1, depth + 1)]
        tm = Timer(torch, stream, dev, g, ctx)
        K = max(3, args.cfg_steps // 2)
        levels = []
        for d in range(0, depth + 1):
            R = built[d]
            n_b = 1 if d == 0 else 1 << (d - 1)
            kernel_bytes, level_bytes = algorithmic_bytes(R, F, wb, B, n_b, 0 if d == 0 else n_b, root=d == 0)
            step = root_step if d == 0 else (lambda d=d: adv_step(d))
            ms, launches, _ = tm.run(step, K, warmup=2)
            _, _, kern = tm.run(step, K, warmup=1, profile_kernels=KERNELS)
            e = level_summary(ms, R * F, level_bytes, peak)
            e.update({"level": d, "rows_built": R, "nodes_built": n_b, "nodes_derived": 0 if d == 0 else n_b,
                      "kernels_ms_per_launch": kern, "gpu_launches_per_step": launches / len(ms),
                      "roofline": roofline_obj("k_hist_u8", kernel_bytes, kern.get("k_hist_u8"), peak, peak_kind)})
            if d > 0:
                pms, _, _ = tm.run(lambda d=d: part_step(d), K, warmup=1)
                e["partition_ms"] = statistics.mean(pms)
                _, _, pk = tm.run(lambda d=d: part_step(d), K, warmup=0, profile_kernels=KERNELS)
                e["partition_kernels_ms_per_launch"] = pk
            levels.append(e)
        tms, tl, _ = tm.run(tree_step, max(2, K // 2), warmup=1)
        assert sess.sync() == 0
        sess.close()
        del tm, lvl
    out["levels"] = levels
    t_tree = statistics.mean(tms)
    tree_entries = sum(built) * F
    out["tree"] = {"ms_per_tree": t_tree, "entries_per_tree": tree_entries, "value": tree_entries / (t_tree / 1e3),
                   "unit": UNIT, "gpu_launches_per_tree": tl / len(tms),
                   "note": "root + 7 x (partition + level step), L2 flushed before each tree only"}
    torch.cuda.empty_cache()
    out["cpu_baseline"] = dense_cpu_baselines(w, args.cpu_budget)
    return out


def dense_cpu_baselines(w, budget_s, S=120_000, pairs=8):
    """CPU baselines of the dense tree on bounded samples: level 0 restricted to the first S rows, and
    `pairs` sibling pairs shaped like level 7's (nodes of N / 128 rows drawn at random from the matrix)."""
    N = w.n_rows
    rng = np.random.default_rng(synth.SEED_BASE + 3)
    sub_w = synth.Workload(name=w.name, n_rows=N, n_features=w.n_features, width=w.width, n_bins=w.n_bins,
                           sentinel=w.sentinel, bins=w.bins, gpair=w.gpair, levels={}, target_depth=0)
    lv0 = synth.Level(depth=0, rows=np.arange(S, dtype=np.int32), offsets=np.array([0, S], np.int64))
    n_nodes = 2 * pairs
    M = n_nodes * (N // 128)
    ids = np.sort(rng.choice(N, size=M, replace=False)).astype(np.int32)
    lv7 = synth.level_from_ids(rng.integers(0, n_nodes, size=M), 7, n_nodes)
    # level_from_ids groups positions 0..M-1 by node; map them to the drawn row ids (ascending in a node)
    lv7.rows = ids[lv7.rows]
    lv7.built_rows = ids[lv7.built_rows]
    parent_rows = (lv7.rows, lv7.offsets[::2].copy())
    shape7 = f"{pairs} sibling pairs shaped like level 7's ({N // 128} random rows per node)"
    cpu = {}
    ov0, s0, _ = cpu_oracle_timing(sub_w, budget_s=budget_s / 2, lv=lv0)
    ov7, s7, _ = cpu_oracle_timing(sub_w, budget_s=budget_s / 2, lv=lv7, parent_rows=parent_rows)
    cpu["oracle_level0"] = {"value": ov0, "unit": UNIT, "cores": 1, "kind": "oracle",
                            "sample": f"level 0 restricted to the first {S} rows: {s0}"}
    cpu["oracle_level7"] = {"value": ov7, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"{shape7}: {s7}"}
    o0 = cpu_openmp_timing(sub_w, budget_s=budget_s / 2, lv=lv0)
    o7 = cpu_openmp_timing(sub_w, budget_s=budget_s / 2, lv=lv7, parent_rows=parent_rows)
    if "sample" in o0:
        o0["sample"] = f"level 0 restricted to the first {S} rows: {o0['sample']}"
    if "sample" in o7:
        o7["sample"] = f"{shape7}: {o7['sample']}"
    cpu["openmp_level0"], cpu["openmp_level7"] = o0, o7
    return cpu


def run_gpu(args, rank, world, local_rank):
    import torch

    import histogram_construction_gb300 as g
    from histogram_construction_gb300.session import Session

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    w = synth.make(args.workload)
    sg, sh = scales_for(w)
    par, lv = level_plan(w)
    B = w.n_bins + 1
    entries, R, n_b, n_p, kernel_bytes, level_bytes = entries_and_bytes(w, lv, B)
    stream = torch.cuda.Stream(dev)
    prop = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(prop, "L2_cache_size", 0) or 0) or (129 << 20)
    hist_kernel = "k_hist_u8" if w.width == 1 else "k_hist_u16"
    with torch.cuda.stream(stream):
        sess = Session(local_rank, stream=stream)
        sess.upload_bins(torch.from_numpy(w.bins).to(dev), w.n_bins, w.sentinel)
        gp_d = torch.from_numpy(w.gpair).to(dev)
        sess.begin_tree(gp_d, sg, sh)
        if lv.depth > 0:
            hp = sess.build_level(torch.from_numpy(par.rows).to(dev), torch.from_numpy(par.offsets).to(dev))
            rows_d = torch.from_numpy(lv.built_rows).to(dev)
            offs_d = torch.from_numpy(lv.built_offsets).to(dev)
            hs = sess.hist_tensor(n_b)
            large = torch.empty_like(hs)
            so = torch.empty((n_p, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)
            lo = torch.empty_like(so)
            prm = g.params(1.0, 0.0, 0.0)
        else:
            rows_d = None
            offs_d = torch.from_numpy(lv.offsets).to(dev)
            hs = sess.hist_tensor(1)
            so = torch.empty((1, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)
            prm = g.params(1.0, 0.0, 0.0)
        flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
        ctx = sess.ctx

        def step():
            if lv.depth > 0:
                if args.path == "fused":
                    sess.check(g.gbt_level_step(ctx, rows_d, offs_d, n_p, hp, None, hs, large, prm, so, lo))
                else:
                    sess.check(g.gbt_build_level(ctx, rows_d, offs_d, n_b, hs))
                    sess.check(g.gbt_subtract_and_find(ctx, hp, None, hs, large, n_p, prm, so, lo))
            else:
                sess.check(g.gbt_build_level(ctx, None, offs_d, 1, hs))
                sess.check(g.gbt_find_splits(ctx, hs, 1, prm, so))

        def flush(i):
            flush_buf.fill_(i & 0xFF)

        for i in range(args.warmup):
            flush(i)
            step()
        assert sess.sync() == 0
        barrier()

        kernel_names = [hist_kernel, "k_level_plan", "k_subtract_find", "k_level_finish", "k_finalize", "k_find"]

        def timed_pass(profile, flush_l2=True):
            """K steps, each bracketed by CUDA events on the launching stream (flush outside the events)."""
            g.gbt_profile_enable(ctx, profile)
            g.gbt_profile_read(ctx)  # forget earlier records
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(args.steps)]
            l0 = g.gbt_kernel_launches(ctx)
            barrier()
            t0 = time.perf_counter()
            for i in range(args.steps):
                if flush_l2:
                    flush(i)
                ev[i][0].record(stream)
                step()
                ev[i][1].record(stream)
            barrier()
            wall = time.perf_counter() - t0
            launches = g.gbt_kernel_launches(ctx) - l0
            ms = [a.elapsed_time(b) for a, b in ev]
            snap = {}
            if profile:
                for name in kernel_names:
                    _, t, n = g.gbt_profile_read(ctx, name)
                    snap[name] = (t, n)
                g.gbt_profile_enable(ctx, False)
            return ms, wall, launches, snap

        clocks = ClockSampler(local_rank).start() if rank == 0 else None
        ms, wall, launches, _ = timed_pass(False)
        # second pass with per-kernel events: device time of each kernel over K steps
        ms_prof, _, _, snap = timed_pass(True)
        clk = clocks.stop() if clocks is not None else None
        # warm-L2 pass (reported second)
        ms_warm, _, _, _ = timed_pass(False, flush_l2=False)
        assert sess.sync() == 0

        # ---------------------------------------------------------------- oblivious level split (optional)
        obl = None
        if args.oblivious and lv.depth > 0:
            lvl_h = torch.cat([hs, large])  # every node of the level
            n_lvl = lvl_h.shape[0]
            lo_out = torch.empty((1, g.SPLIT_BYTES), dtype=torch.uint8, device=dev)
            for i in range(3):
                sess.check(g.gbt_find_level_split(ctx, lvl_h, n_lvl, prm, lo_out))
            obl_ms = []
            for i in range(args.steps):
                flush(i)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                sess.check(g.gbt_find_level_split(ctx, lvl_h, n_lvl, prm, lo_out))
                b.record(stream)
                b.synchronize()
                obl_ms.append(a.elapsed_time(b))
            assert sess.sync() == 0
            obl_bytes = n_lvl * w.n_features * B * 16
            obl_t = statistics.median(obl_ms)
            obl = {"nodes": n_lvl, "ms_per_call": obl_t, "algorithmic_bytes": obl_bytes,
                   "achieved_gbs": obl_bytes / (obl_t / 1e3) / 1e9}

        # ---------------------------------------------------------------- float-cell level (optional)
        f64 = None
        if args.f64 and lv.depth > 0:
            hp64 = sess.build_level_f64(gp_d, torch.from_numpy(par.rows).to(dev), torch.from_numpy(par.offsets).to(dev))
            hs64 = torch.empty((n_b, w.n_features, B, 2), dtype=torch.float64, device=dev)
            large64 = torch.empty_like(hs64)
            so64 = torch.empty_like(so)
            lo64 = torch.empty_like(so)

            def step64():
                sess.check(g.gbt_build_level_f64(ctx, gp_d, rows_d, offs_d, n_b, hs64))
                sess.check(g.gbt_subtract_siblings_f64(ctx, hp64, None, hs64, large64, n_p))
                sess.check(g.gbt_find_splits_f64(ctx, hs64, n_b, prm, so64))
                sess.check(g.gbt_find_splits_f64(ctx, large64, n_p, prm, lo64))

            for i in range(3):
                flush(i)
                step64()
            assert sess.sync() == 0
            f64_ms = []
            for i in range(args.steps):
                flush(i)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step64()
                b.record(stream)
                b.synchronize()
                f64_ms.append(a.elapsed_time(b))
            assert sess.sync() == 0
            f64_t = statistics.median(f64_ms)
            f64 = {"ms_per_step": f64_t, "entries_per_s": entries / (f64_t / 1e3),
                   "note": "same level in double cells of the unquantised float32 gpair"}
            del hp64, hs64, large64

        # ---------------------------------------------------------------- multi-output level (optional)
        multi = None
        if args.multi > 0 and w.width == 1:
            k = args.multi
            gpm = synth.gpair_multi(args.workload, w.n_rows, k)
            msg, msh = [], []
            for t in range(k):
                a_, b_ = synth.fixed_point_scales(gpm[:, t, :])
                msg.append(a_)
                msh.append(b_)
            sess.begin_tree_multi(torch.from_numpy(gpm).to(dev), msg, msh)
            m_rows = rows_d if lv.depth > 0 else None
            m_offs = offs_d
            hm = torch.empty((k, n_b, w.n_features, B, 2), dtype=torch.int64, device=dev)

            def step_multi():
                sess.check(g.gbt_build_level_multi(ctx, m_rows, m_offs, n_b, hm))

            for i in range(3):
                flush(i)
                step_multi()
            assert sess.sync() == 0
            m_ms = []
            g.gbt_profile_enable(ctx, True)
            g.gbt_profile_read(ctx)
            for i in range(args.steps):
                flush(i)
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                step_multi()
                b.record(stream)
                b.synchronize()
                m_ms.append(a.elapsed_time(b))
            mk = {}
            for name in ("k_level_plan", "k_hist_u8_multi", "k_finalize_multi"):
                _, t_, n_ = g.gbt_profile_read(ctx, name)
                if n_:
                    mk[name] = t_ / n_
            g.gbt_profile_enable(ctx, False)
            assert sess.sync() == 0
            # bins once per target group of four, (row id, k pairs) per row, k partial images written
            m_kbytes = R * w.n_features * ((k + 3) // 4) + R * (4 + 8 * k) + k * n_b * w.n_features * B * 8
            m_t = statistics.median(m_ms)
            hk = mk.get("k_hist_u8_multi")
            multi = {"targets": k, "ms_per_call": m_t, "target_entries_per_s": k * entries / (m_t / 1e3),
                     "kernels_ms_per_launch": mk, "hist_kernel_algorithmic_bytes": m_kbytes,
                     "hist_kernel_achieved_gbs": (m_kbytes / (hk / 1e3) / 1e9) if hk else None,
                     "note": "gbt_build_level_multi on the level's built nodes: k int64 histograms, one bin pass"}
            del hm

        # ---------------------------------------------------------------- e2e through host buffers
        e2e = None
        if lv.depth > 0:
            rows_h = torch.from_numpy(lv.built_rows).pin_memory()
            offs_h = torch.from_numpy(lv.built_offsets).pin_memory()
            so_h = torch.empty((n_p, g.SPLIT_BYTES), dtype=torch.uint8).pin_memory()
            lo_h = torch.empty_like(so_h).pin_memory()
            h2d = rows_h.numel() * 4 + offs_h.numel() * 8
            d2h = 2 * n_p * g.SPLIT_BYTES

            def step_e2e():
                sess.check(g.gbt_level_step(ctx, rows_h, offs_h, n_p, hp, None, hs, large, prm, so_h, lo_h))
        else:
            gp_h = torch.from_numpy(w.gpair).pin_memory()
            offs_h = torch.from_numpy(lv.offsets).pin_memory()
            so_h = torch.empty((1, g.SPLIT_BYTES), dtype=torch.uint8).pin_memory()
            h2d = gp_h.numel() * 4 + offs_h.numel() * 8
            d2h = g.SPLIT_BYTES

            def step_e2e():
                sess.check(g.gbt_begin_tree(ctx, gp_h, sg, sh))
                sess.check(g.gbt_build_level(ctx, None, offs_h, 1, hs))
                sess.check(g.gbt_find_splits(ctx, hs, 1, prm, so_h))
        for i in range(3):
            flush(i)
            step_e2e()
            sess.check(sess.sync())
        e2e_ms = []
        for i in range(args.steps):
            flush(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_e2e()
            b.record(stream)
            b.synchronize()  # the host reads the step's result
            e2e_ms.append(a.elapsed_time(b))
        assert sess.sync() == 0
        e2e = {"value": entries / (statistics.mean(e2e_ms) / 1e3) * world, "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}
        sess.close()
        del flush_buf

    total_ms, e2e_value = aggregate_ranks(sum(ms), e2e["value"], world, dist, dev)
    e2e["value"] = e2e_value
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak, peak_kind = _peaks()
    value = job_throughput(world, args.steps, entries, total_ms)
    hk_ms, hk_n = snap[hist_kernel]
    hk_avg = hk_ms / max(hk_n, 1) if hk_n else None
    traffic = _profile_traffic(args.workload) if w.width == 1 else None
    step_ms = total_ms / args.steps
    level_entries = int(lv.offsets[-1]) * w.n_features
    level_gbs = level_bytes / (step_ms / 1e3) / 1e9
    cpu_v, cpu_sample, _ = cpu_oracle_timing(w, budget_s=args.cpu_budget)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "median_ms_per_step": statistics.median(ms),
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "int64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "rows_built": R, "features": w.n_features,
                   "bin_bytes": w.width, "slots_per_feature": B, "nodes_built": n_b, "nodes_derived": n_p,
                   "entries_per_step": entries, "l2": f"flushed before every step ({2 * l2 >> 20} MiB write)",
                   "path": "gbt_level_step" if args.path == "fused" else "gbt_build_level + gbt_subtract_and_find",
                   "parallelism": f"replicas{world}"},
        "roofline": roofline_obj(hist_kernel, kernel_bytes, hk_avg, peak, peak_kind, traffic),
        "level_roofline": {"algorithmic_bytes_per_step": level_bytes, "achieved_gbs": level_gbs,
                           "frac": level_gbs / peak, "peak": peak},
        "kernels_ms_per_launch": {k: (v[0] / max(v[1], 1)) for k, v in snap.items() if v[1]},
        "profiled_pass_ms_per_step": sum(ms_prof) / len(ms_prof),
        "warm_l2": {"ms_per_step": sum(ms_warm) / len(ms_warm),
                    "value": world * entries / (sum(ms_warm) / len(ms_warm) / 1e3)},
        # every row of the level (built and derived siblings) x F over the same step time
        "effective": {"entries_per_step": level_entries,
                      "value": world * level_entries / (step_ms / 1e3)},
        "e2e": e2e,
        "gpu_launches": int(launches),
        "clocks": clk,
        "cpu_baseline": {"value": cpu_v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": cpu_sample},
        "cpu_baseline_openmp": cpu_openmp_timing(w, budget_s=args.cpu_budget),
        "host": {"nproc": os.cpu_count()},
        "wall_s_timed": wall,
    }
    if obl is not None:
        obl["frac"] = obl["achieved_gbs"] / peak
        line["oblivious_split"] = obl
    if f64 is not None:
        line["float_cells"] = f64
    if multi is not None:
        multi["hist_kernel_frac"] = (multi["hist_kernel_achieved_gbs"] / peak
                                     if multi["hist_kernel_achieved_gbs"] else None)
        line["multi_output"] = multi
    if args.per_config:
        torch.cuda.empty_cache()
        per = {}
        clocks = ClockSampler(local_rank).start()
        for name in [c for c in args.configs.split(",") if c and c != args.workload]:
            if name == "dense":
                per[name] = run_dense_tree(torch, g, dev, stream, args, peak, peak_kind)
            else:
                per[name] = run_config_level(name, torch, g, dev, stream, args, peak, peak_kind)
        per["clocks"] = clocks.stop()
        line["per_config"] = per
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = synth.make(args.workload)
    par, lv = level_plan(w)
    B = w.n_bins + 1
    entries, R, n_b, n_p, kernel_bytes, level_bytes = entries_and_bytes(w, lv, B)
    v, sample, per = cpu_oracle_timing(w, budget_s=args.ref_budget, steps=args.steps, warmup=args.warmup)
    line = {
        "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(per), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int64", "data": "synthetic",
        "config": {"workload": WORKLOAD_TEXT[args.workload], "rows_built": R, "features": w.n_features,
                   "bin_bytes": w.width, "slots_per_feature": B, "nodes_built": n_b, "nodes_derived": n_p,
                   "entries_per_step": entries, "parallelism": "serial CPU oracle"},
        "impl": "reference",
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOAD_TEXT), default="level5")
    ap.add_argument("--path", choices=["fused", "unfused"], default="fused")
    ap.add_argument("--f64", action="store_true",
                    help="also time the level in float-cell mode (double cells; reported under float_cells)")
    ap.add_argument("--oblivious", action="store_true",
                    help="also time gbt_find_level_split on the level's histograms (reported under oblivious_split)")
    ap.add_argument("--multi", type=int, default=0, metavar="K",
                    help="also time gbt_build_level_multi with K targets on the level (u8; reported under multi_output)")
    ap.add_argument("--per-config", dest="per_config", action="store_true", default=True,
                    help="also measure the other workloads (default)")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false")
    ap.add_argument("--configs", default=",".join(PER_CONFIG), help="workloads of per_config, comma-separated")
    ap.add_argument("--cfg-steps", type=int, default=20, help="timed steps per per_config workload")
    ap.add_argument("--cpu-budget", type=float, default=4.0, help="seconds of CPU time per cpu_baseline sample")
    ap.add_argument("--ref-budget", type=float, default=90.0, help="seconds of oracle time for --impl reference")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_gpu(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
