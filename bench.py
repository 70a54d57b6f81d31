#!/usr/bin/env python
"""Benchmark of the level histogram path: binned entries per second per level on GB300.

One step = one tree level of the workload through gbt_level_step: the
histograms of the smaller siblings (level plan + histogram kernel), sibling
subtraction and split find for both siblings of every pair (level-finish
kernel). ``--path unfused`` times gbt_build_level + gbt_subtract_and_find
instead. Inputs are resident in HBM when the timed region starts; L2 is
flushed (a write larger than L2) before every step, outside the step's CUDA
events.

Prints one JSON line (rank 0). ``--impl reference`` times the serial CPU oracle
on the same workload instead (rank 0 only).
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
}


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


def entries_and_bytes(w, lv, B):
    """Units of one step and the algorithmic HBM bytes (per level and for the histogram kernel alone)."""
    F, wb = w.n_features, w.width
    if lv.depth == 0:
        R = int(lv.offsets[-1])
        n_b, n_p = 1, 0
    else:
        R = int(lv.built_offsets[-1])
        n_b = n_p = len(lv.small)
    entries = R * F
    # histogram kernel: read the bins and (row id, qg, qh) of every built row, write each
    # built node's exact 32-bit partial (the least it can hand on)
    kernel_bytes = R * F * wb + R * 12 + n_b * F * B * 8
    # whole level (fused path): bins + row ids/gradients, read parents, write small and large
    level_bytes = R * F * wb + R * 12 + 3 * n_p * F * B * 16 if n_p else R * F * wb + R * 8 + n_b * F * B * 16
    return entries, R, n_b, n_p, kernel_bytes, level_bytes


def scales_for(w):
    """The workload's fixed-point scales (equal to gbt_suggest_scales on the same data; tests/test_abi.py)."""
    return synth.fixed_point_scales(w.gpair)


# ----------------------------------------------------------------------------- CPU oracle leg
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


def cpu_oracle_timing(w, budget_s=10.0, steps=None, warmup=0):
    """Time the oracle as it stands (1 thread). Returns (entries/s, sample text, per-step seconds)."""
    import oracle
    sg, sh = scales_for(w)
    q, _ = oracle.quantise(w.gpair, sg, sh)
    par, lv = level_plan(w)
    parent_hist = None
    if par is not None:
        parent_hist, _ = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, par.rows, par.offsets)
    # calibrate one full step
    t0 = time.perf_counter()
    e_full = oracle_level(oracle, w, q, lv, parent_hist, sg, sh)
    t_full = time.perf_counter() - t0
    node_slice = None
    if steps is not None:
        n_total = steps + warmup
        if lv.depth > 0 and n_total * t_full > budget_s:
            frac = budget_s / (n_total * t_full)
            node_slice = max(1, int(len(lv.small) * frac))
        for _ in range(warmup):
            oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice)
        ent, t0 = 0, time.perf_counter()
        per = []
        for _ in range(steps):
            ts = time.perf_counter()
            ent += oracle_level(oracle, w, q, lv, parent_hist, sg, sh, node_slice)
            per.append(time.perf_counter() - ts)
        dt = time.perf_counter() - t0
        n_nodes = len(lv.small) if lv.depth > 0 else 1
        sample = (f"{steps} steps of {'the full level' if node_slice is None else f'the first {node_slice} of {n_nodes} built nodes'}"
                  f" ({ent // steps} entries per step)")
        return ent / dt, sample, per
    reps, ent, dt = 1, e_full, t_full
    while dt < budget_s:
        t0 = time.perf_counter()
        ent += oracle_level(oracle, w, q, lv, parent_hist, sg, sh)
        dt += time.perf_counter() - t0
        reps += 1
    return ent / dt, f"the full level ({e_full} entries: build, subtract, split find) x {reps} repetitions", None


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
                _, a_, b_ = g.gbt_suggest_scales(0, float(np.abs(gpm[:, t, 0]).max()), float(np.abs(gpm[:, t, 1]).max()))
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

    total_ms, e2e_value = aggregate_ranks(sum(ms), e2e["value"], world, dist, dev)
    e2e["value"] = e2e_value
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    peak, peak_kind = _peaks()
    value = job_throughput(world, args.steps, entries, total_ms)
    hk_ms, hk_n = snap[hist_kernel]
    hk_avg = hk_ms / max(hk_n, 1)
    achieved = kernel_bytes / (hk_avg / 1e3) / 1e9 if hk_n else None
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
        "roofline": {"bound": "hbm", "kernel": hist_kernel, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": (achieved / peak) if achieved else None, "traffic": traffic,
                     "algorithmic_bytes_per_launch": kernel_bytes, "avg_launch_ms": hk_avg,
                     "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"},
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
        "wall_s_timed": wall,
    }
    if obl is not None:
        peak_v, _ = _peaks()
        obl["frac"] = obl["achieved_gbs"] / peak_v
        line["oblivious_split"] = obl
    if f64 is not None:
        line["float_cells"] = f64
    if multi is not None:
        multi["hist_kernel_frac"] = (multi["hist_kernel_achieved_gbs"] / peak
                                     if multi["hist_kernel_achieved_gbs"] else None)
        line["multi_output"] = multi
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
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle time for cpu_baseline")
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
