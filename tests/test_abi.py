"""The C-ABI library builds, loads without a GPU and exports every symbol its header declares."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "gbthist.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gbt_[a-z0-9_]+)\s*\(", text)))


def test_library_builds_and_exports_header_symbols():
    import histogram_construction_gb300 as g
    path = g.lib_path()
    g.lib()  # builds with nvcc if needed
    raw = ctypes.CDLL(path)
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(raw, n), f"{n} declared in gbthist.h but not exported"
    assert set(names) == set(g.EXPORTS)


def test_split_struct_layout_matches_header():
    import histogram_construction_gb300 as g
    assert ctypes.sizeof(g.GbtSplit) == 56
    assert g.GbtSplit.gain.offset == 16 and g.GbtSplit.g_left.offset == 24


@pytest.mark.parametrize("rows,mg,mh", [(0, 5.3, 1.0), (65536, 1.0, 0.25), (1, 3.0, 3.0), (10_000_000, 4.0, 1.0)])
def test_suggest_scales_is_largest_power_of_two_within_bound(rows, mg, mh):
    import math

    import histogram_construction_gb300 as g
    st, sg, sh = g.gbt_suggest_scales(rows, mg, mh)
    assert st == 0
    r = max(rows if rows > 0 else 65536, 1024)  # documented floor of 1024 rows per partial
    for m, s in ((mg, sg), (mh, sh)):
        assert math.log2(s) == int(math.log2(s))
        assert m * s * r <= 2 ** 31 - 1
        assert m * (2 * s) * r > 2 ** 31 - 1


@pytest.mark.parametrize("name", ["root", "level5", "u16miss"])
def test_workload_scales_equal_the_library_suggestion(name):
    """The benchmark and tests run every workload with synth.fixed_point_scales (so its CPU legs never
    load the library); that is exactly what gbt_suggest_scales returns for the same data."""
    import numpy as np

    import histogram_construction_gb300 as g
    import synth
    rng = np.random.default_rng(7)
    for gp in (synth.make(name, n_rows=5000, n_features=3).gpair,
               (rng.standard_normal((100, 2)) * [1e-3, 7e4]).astype(np.float32),
               np.zeros((4, 2), np.float32)):
        st, sg, sh = g.gbt_suggest_scales(0, float(np.abs(gp[:, 0]).max()), float(np.abs(gp[:, 1]).max()))
        assert st == 0
        assert synth.fixed_point_scales(gp) == (sg, sh)


def test_suggest_scales_rejects_bad_input():
    import histogram_construction_gb300 as g
    assert g.gbt_suggest_scales(0, float("nan"), 1.0)[0] == g.GBT_ERR_INVALID_ARG
    assert g.gbt_suggest_scales(0, -1.0, 1.0)[0] == g.GBT_ERR_INVALID_ARG


def test_create_without_device_fails_cleanly():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    import histogram_construction_gb300 as g
    st, h = g.gbt_create(0)
    assert st != 0 and h is None
    assert g.gbt_destroy(None) == 0
