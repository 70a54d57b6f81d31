"""GPU parity of the float-cell mode against the serial oracle.

The GPU follows the pages' precision scheme: float shared-memory cells per
chunk of at most 32768 rows, merged across chunks in double; the oracle sums
every cell serially in double. Two bars:
  * dyadic gpair (every g, h a multiple of 2^-6 with |g| < 4): a chunk's float
    sums stay below 2^17 and so are exact, as are the double merges and the
    oracle's sums; histograms, subtraction and splits (gains included) are
    compared bit for bit;
  * generic float gpair: a float sum of m values in any order is within
    gamma_24(m - 1) * (sum of |x|) of the exact sum (gamma_p(k) = k 2^-p /
    (1 - k 2^-p)); the double merge and the oracle's serial double sum add
    gamma_53 terms over the node's n rows. The test bounds each cell by
    (gamma_24(m - 1) + 3 n 2^-53) * (sum of |x| over the cell), m = min(n,
    32768). The split found on the GPU's histogram is checked against the
    oracle's split of that same histogram: the same gain within 1e-12
    relative, and the same (feature, bin, direction) unless the chosen
    candidate's own oracle gain is that close to the best.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

U = 2.0 ** -53


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g
    from histogram_construction_gb300.session import SPLIT_F64_DTYPE, Session, splits_to_numpy
    g.lib()
    return g, Session, lambda t: splits_to_numpy(t, SPLIT_F64_DTYPE)


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    return o


CHUNK = 32768


def dyadic(gp):
    """g to a multiple of 2^-6 in (-4, 4), h to a positive multiple of 2^-6."""
    out = np.empty_like(gp)
    out[:, 0] = np.clip(np.round(gp[:, 0] * 64.0), -255.0, 255.0) / 64.0
    out[:, 1] = np.maximum(np.round(gp[:, 1] * 64.0), 1.0) / 64.0
    return out


def assert_cells_close(got, ref, ab, offsets, where):
    n = np.diff(np.asarray(offsets, dtype=np.int64)).astype(np.float64)
    m = np.minimum(n, CHUNK)
    k = np.maximum(m - 1.0, 0.0) * 2.0 ** -24
    tol = ((k / (1.0 - k)) + 3.0 * n * U)[:, None, None, None] * ab
    err = np.abs(got - ref)
    bad = err > tol
    assert not bad.any(), f"{where}: {int(bad.sum())} cells off, worst {float((err - tol).max())}"
    # the per-cell bar of the float mode: |a - b| <= 1e-5 * (sum of |x| over the cell)
    bad = err > 1e-5 * ab
    assert not bad.any(), f"{where}: {int(bad.sum())} cells beyond 1e-5 of their absolute sum"


def assert_splits_bitwise(got, ref, where):
    for k in ("feature", "bin", "default_left"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{where} {k}")
    for k in ("gain", "g_left", "h_left", "g_right", "h_right"):
        np.testing.assert_array_equal(got[k].view(np.int64), ref[k].view(np.int64), err_msg=f"{where} {k}")


def assert_splits_close(got, ref, hist, n_bins, lam, gamma, mcw, oracle, where):
    """got: GPU splits of `hist`; ref: oracle splits of the same histogram."""
    for n in range(got.shape[0]):
        if ref["feature"][n] < 0:
            assert got["feature"][n] < 0 or not np.isfinite(got["gain"][n]), f"{where} node {n}"
            continue
        g, r = float(got["gain"][n]), float(ref["gain"][n])
        assert abs(g - r) <= 1e-12 * max(1.0, abs(r)), f"{where} node {n}: gain {g} vs {r}"
        same = (got["feature"][n], got["bin"][n], got["default_left"][n]) == \
               (ref["feature"][n], ref["bin"][n], ref["default_left"][n])
        if not same:
            # another candidate within rounding of the best: its own oracle gain must be that close too
            f, t, d = int(got["feature"][n]), int(got["bin"][n]), int(got["default_left"][n])
            hf = hist[n, f]
            G, H = hf[:, 0].sum(), hf[:, 1].sum()
            GL = hf[:t + 1, 0].sum() + (hf[n_bins, 0] if d else 0.0)
            HL = hf[:t + 1, 1].sum() + (hf[n_bins, 1] if d else 0.0)
            alt = oracle.gain(GL, HL, G - GL, H - HL, G, H, lam, gamma)
            assert abs(alt - r) <= 1e-12 * max(1.0, abs(r)), f"{where} node {n}: chose {(f, t, d)} gain {alt} vs {r}"
        for k in ("g_left", "h_left", "g_right", "h_right"):
            a, b = float(got[k][n]), float(ref[k][n])
            if same:
                assert abs(a - b) <= 1e-9 * max(1.0, abs(b)), f"{where} node {n} {k}: {a} vs {b}"


def level_pair(sess, oracle, w, depth, gp, lam=1.0, gamma=0.0, mcw=0.0, exact=True, device_gp=True):
    """Parents at depth-1 (all their rows), the smaller siblings at depth, subtract, find; compare everything."""
    par, lv = w.levels[depth - 1], w.levels[depth]
    gpa = torch.from_numpy(gp).cuda() if device_gp else gp
    hp = sess.build_level_f64(gpa, par.rows, torch.from_numpy(par.offsets).cuda())
    hs = sess.build_level_f64(gpa, lv.built_rows, lv.built_offsets)
    large = sess.subtract_f64(hp, hs)
    so = sess.find_splits_f64(hs, lam, gamma, mcw)
    lo = sess.find_splits_f64(large, lam, gamma, mcw)
    assert sess.sync() == 0
    ref_hp, ab_p, st = oracle.build_hist_f64(w.bins, w.n_bins, w.sentinel, gp, par.rows, par.offsets)
    assert st == oracle.OK
    ref_hs, ab_s, st = oracle.build_hist_f64(w.bins, w.n_bins, w.sentinel, gp, lv.built_rows, lv.built_offsets)
    assert st == oracle.OK
    g_hp, g_hs, g_large = hp.cpu().numpy(), hs.cpu().numpy(), large.cpu().numpy()
    if exact:
        np.testing.assert_array_equal(g_hp, ref_hp, err_msg="parent hist")
        np.testing.assert_array_equal(g_hs, ref_hs, err_msg="small hist")
    else:
        assert_cells_close(g_hp, ref_hp, ab_p, par.offsets, "parent hist")
        assert_cells_close(g_hs, ref_hs, ab_s, lv.built_offsets, "small hist")
    # subtraction: one rounding per cell on the GPU's own operands, so bit-exact against the oracle's
    ref_large, st = oracle.subtract_f64(g_hp, None, g_hs)
    assert st == oracle.OK
    np.testing.assert_array_equal(g_large, ref_large, err_msg="large hist")
    ref_large_o, _ = oracle.subtract_f64(ref_hp, None, ref_hs)
    for name, h, s, h_o in (("small", g_hs, so, ref_hs), ("large", g_large, lo, ref_large_o)):
        ref, st = oracle.find_splits_f64(h, w.n_bins, lam, gamma, mcw)
        assert st == oracle.OK
        got = gb_split(s)
        if exact:
            assert_splits_bitwise(got, ref, f"{name} splits")
        else:
            assert_splits_close(got, ref, h, w.n_bins, lam, gamma, mcw, oracle, f"{name} splits")
            # end to end against the oracle's own histograms: best gains within 1e-5 relative
            ref_o, _ = oracle.find_splits_f64(h_o, w.n_bins, lam, gamma, mcw)
            fin = np.isfinite(ref_o["gain"])
            np.testing.assert_array_equal(np.isfinite(got["gain"]), fin, err_msg=f"{name} valid nodes")
            # 1e-5 relative to the gain's own terms (the gain is a difference of them)
            r = ref_o[fin]
            G, H = r["g_left"] + r["g_right"], r["h_left"] + r["h_right"]
            mag = 0.5 * (r["g_left"] ** 2 / (r["h_left"] + lam) + r["g_right"] ** 2 / (r["h_right"] + lam)
                         + G ** 2 / (H + lam)) + abs(gamma)
            err = np.abs(got["gain"][fin] - r["gain"])
            assert (err <= 1e-5 * np.maximum(np.abs(r["gain"]), mag)).all(), f"{name} gains vs the oracle's histograms"
    return g_hp, g_hs, g_large


gb_split = None


@pytest.fixture(autouse=True)
def _split_reader(gb):
    global gb_split
    gb_split = gb[2]


def test_level5_dyadic_bitexact(gb, oracle):
    g, Session, _ = gb
    w = synth.make("level5", n_rows=120_000, n_features=70, depth=3)
    gp = dyadic(w.gpair)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        for d in (1, 3):
            level_pair(s, oracle, w, d, gp)
        level_pair(s, oracle, w, 2, gp, lam=0.5, gamma=0.25, mcw=3.0, device_gp=False)
        # lambda < 0 switches the FP32 screen off: every valid candidate is evaluated in double
        level_pair(s, oracle, w, 1, gp, lam=-0.25, mcw=1.0)


def test_chunk_cap_many_full_chunks(gb, oracle, monkeypatch):
    """A load-balance target of 8 items makes every chunk hit the 32768-row cap: multi-chunk double merges
    of full float chunks, and image scratch sized by the cap."""
    g, Session, _ = gb
    w = synth.make("level5", n_rows=300_000, n_features=130, depth=1)
    gp = dyadic(w.gpair)
    monkeypatch.setenv("GBT_TARGET_ITEMS", "8")
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        offs = np.array([0, w.n_rows], dtype=np.int64)
        h = s.build_level_f64(torch.from_numpy(gp).cuda(), None, offs)
        assert s.sync() == 0
        ref, _, _ = oracle.build_hist_f64(w.bins, w.n_bins, w.sentinel, gp, None, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        level_pair(s, oracle, w, 1, gp)
        level_pair(s, oracle, w, 1, w.gpair, exact=False)


def test_level5_float_within_rounding(gb, oracle):
    g, Session, _ = gb
    w = synth.make("level5", n_rows=150_000, n_features=45, depth=3)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        for d in (1, 2, 3):
            level_pair(s, oracle, w, d, w.gpair, exact=False)


def test_root_identity_rows(gb, oracle):
    """rows = None (identity) for the root; one node; tiny feature count."""
    g, Session, _ = gb
    w = synth.make("root")
    gp = dyadic(w.gpair)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        offs = np.array([0, w.n_rows], dtype=np.int64)
        h = s.build_level_f64(torch.from_numpy(gp).cuda(), None, offs)
        sp = s.find_splits_f64(h, 1.0, 0.0, 1.0)
        assert s.sync() == 0
        ref, _, st = oracle.build_hist_f64(w.bins, w.n_bins, w.sentinel, gp, None, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        rs, _ = oracle.find_splits_f64(ref, w.n_bins, 1.0, 0.0, 1.0)
        assert_splits_bitwise(gb_split(sp), rs, "root")


def test_wide_ragged_feature_groups(gb, oracle):
    """4133 features: 130 float-cell feature groups of 32, the last holding 5; 2 KB-wide mirror rows."""
    g, Session, _ = gb
    w = synth.make("wide", n_rows=8192, n_features=4133)
    gp = dyadic(w.gpair)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        level_pair(s, oracle, w, w.target_depth, gp)


def test_u16_missing(gb, oracle):
    """u16 bins, 4096 bins + missing slot, 40% missing (summed in registers per lane)."""
    g, Session, _ = gb
    w = synth.make("u16miss", n_rows=60_000, n_features=11, depth=3)
    gp = dyadic(w.gpair)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        level_pair(s, oracle, w, 3, gp)
        level_pair(s, oracle, w, 2, w.gpair, exact=False, mcw=1.0)


def test_empty_nodes_and_clamp(gb, oracle):
    g, Session, _ = gb
    w = synth.make("level5", n_rows=20_000, n_features=9, depth=1)
    gp = dyadic(w.gpair)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        rows = w.levels[1].rows
        n1 = int(w.levels[1].offsets[1])
        offs = np.array([0, 0, n1, n1, len(rows), len(rows)], dtype=np.int64)  # empty nodes 0, 2, 4
        h = s.build_level_f64(gp, rows, offs)
        sp = s.find_splits_f64(h)
        assert s.sync() == 0
        ref, _, _ = oracle.build_hist_f64(w.bins, w.n_bins, w.sentinel, gp, rows, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        got = gb_split(sp)
        assert (got["feature"][[0, 2, 4]] == -1).all() and np.isneginf(got["gain"][[0, 2, 4]]).all()
        assert_splits_bitwise(got, oracle.find_splits_f64(ref, w.n_bins, 1.0, 0.0, 0.0)[0], "empty")
        # clamp: a small sibling whose H exceeds the parent's by rounding-sized amounts
        rng = np.random.default_rng(7)
        par = rng.standard_normal((3, 9, w.n_bins + 1, 2))
        par[..., 1] = np.abs(par[..., 1])
        small = par.copy()
        small[..., 1] += rng.choice([0.0, 1e-13, -1e-13], size=small[..., 1].shape)
        small[..., 0] *= 0.5
        po = np.array([2, 0, 1], dtype=np.int32)
        small_p = small[po]
        d_large = s.subtract_f64(torch.from_numpy(par).cuda(), torch.from_numpy(small_p).cuda(), parent_of=po)
        assert s.sync() == 0
        ref_large, st = oracle.subtract_f64(par, po, small_p)
        assert st == oracle.OK
        gl = d_large.cpu().numpy()
        np.testing.assert_array_equal(gl, ref_large)
        assert (gl[..., 1] >= 0).all() and (gl[..., 1] == 0).any()


def test_level5_full_size(gb, oracle):
    """The full 1M x 100 depth-5 level (16 smaller siblings, 16 parents) in float cells."""
    g, Session, _ = gb
    w = synth.make("level5")
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        level_pair(s, oracle, w, 5, w.gpair, exact=False)


def _dyadic_strip(rng, B, scale_g=1.0, scale_h=1.0):
    g = np.round(rng.standard_normal(B) * 64.0 * scale_g) / 64.0
    h = np.maximum(np.round(rng.uniform(0.0, 1.0, B) * 64.0 * scale_h), 1.0) / 64.0
    return np.stack([g, h], axis=-1)


@pytest.mark.parametrize("lam,gamma,mcw,scale", [(1.0, 0.0, 0.0, 1.0), (0.0, 0.5, 2.0, 1.0), (1.0, 0.0, 1.0, 2.0 ** 20),
                                                 (0.25, 0.0, 0.0, 2.0 ** -8)])
def test_split_find_near_ties(gb, oracle, lam, gamma, mcw, scale):
    """Histograms built to stress the FP32 screen: identical features (exact ties: the smallest feature must win),
    copies perturbed by one 2^-6 step moved between neighbouring bins (gains within ~1e-6 of each other),
    min_child_weight landing exactly on prefix sums, and large or small magnitudes. Dyadic cells: every sum is
    exact, so the GPU must match the oracle bit for bit."""
    g, Session, _ = gb
    rng = np.random.default_rng(11)
    n_bins, F, n_nodes = 255, 37, 3
    B = n_bins + 1
    hist = np.zeros((n_nodes, F, B, 2))
    base = _dyadic_strip(rng, B, scale, scale)
    for n in range(n_nodes):
        for f in range(F):
            st = base.copy()
            if n >= 1 and f % 3:
                k = (f * 7 + n) % (B - 2)
                st[k, 0] += 1.0 / 64.0 * scale
                st[k + 1, 0] -= 1.0 / 64.0 * scale
            hist[n, f] = st
    with Session() as s:
        s.upload_bins(np.zeros((F, 64), dtype=np.uint8), n_bins, 255)
        d = torch.from_numpy(hist).cuda()
        sp = s.find_splits_f64(d, lam, gamma, mcw)
        assert s.sync() == 0
        ref, st = oracle.find_splits_f64(hist, n_bins, lam, gamma, mcw)
        assert st == oracle.OK
        got = gb_split(sp)
        assert_splits_bitwise(got, ref, "near ties")
        assert got["feature"][0] == 0  # exact ties across identical features: the first one wins
