"""The all-core OpenMP CPU baseline computes what the oracle computes (no GPU): its int64 histograms equal
the oracle's bit for bit, and its splits pick the same candidates."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("name,n_rows,n_features,depth", [("level5", 20_000, 37, 3), ("u16miss", 15_000, 9, 3)])
def test_openmp_level_matches_oracle(oracle_mod, name, n_rows, n_features, depth):
    cpu_baseline = pytest.importorskip("cpu_baseline")
    try:
        cpu_baseline.build()
    except Exception as e:  # a toolchain without OpenMP
        pytest.skip(f"OpenMP baseline not buildable here: {e}")
    w = synth.make(name, n_rows=n_rows, n_features=n_features, depth=depth)
    sg, sh = synth.fixed_point_scales(w.gpair)
    q, st = oracle_mod.quantise(w.gpair, sg, sh)
    assert st == oracle_mod.OK
    par, lv = w.levels[depth - 1], w.levels[depth]
    hp, _ = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, par.rows, par.offsets)
    hs, _ = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, lv.built_rows, lv.built_offsets)
    hl, _ = oracle_mod.subtract(hp, None, hs)
    small, large, so, lo = cpu_baseline.level(w.bins, w.n_bins, w.sentinel, q, lv.built_rows, lv.built_offsets, hp,
                                              1.0, 0.0, 0.0, sg, sh)
    np.testing.assert_array_equal(small, hs)
    np.testing.assert_array_equal(large, hl)
    for got, h in ((so, hs), (lo, hl)):
        ref, _ = oracle_mod.find_splits(h, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
        for k in ("feature", "bin", "default_left", "g_left", "h_left"):
            np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
