"""Near ties in the split find: distinct candidates whose double gains differ by 0 to 4 ulps.

The FP32 screen of the split find cannot separate such candidates: both reach the double evaluation,
and the winner must be the one the serial oracle picks ('GBDT engine engineering deep-dive', section 1:
the gain formula; bonsai '9. Parallelism & determinism', 'In bonsai': ties break in serial order).
The cases put the near-tied candidates

  (a) in features of different CTAs of one node (the published bounds and the node threshold decide),
  (b) in more than two features of one CTA (the CTA evaluates its survivors itself),
  (c) at two cuts of one strip without missing mass (the one-direction copy of the scan),
  (d) in the two missing directions of one cut,

with strips staged in shared memory (u8 widths, 256 slots) and read from global memory (4097 slots),
under the fast screen, the checked screen (sums beyond 2^45) and no screen (lambda < 0). Every result
is compared bit for bit with oracle.find_splits, and the oracle's own winner is checked to be the
designed one, so a case that stopped being a near tie would fail here too.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _gains(GL, HL, G, H, lam):
    """The gain of candidates (GL, HL) of a node with totals (G, H), unit scales, gamma = 0, in IEEE double
    in the formula's order (used to choose the cases; the comparison itself is with the oracle)."""
    gl = np.asarray(GL, np.int64).astype(np.float64)
    hl = np.asarray(HL, np.int64).astype(np.float64)
    gr = (np.int64(G) - np.asarray(GL, np.int64)).astype(np.float64)
    hr = (np.int64(H) - np.asarray(HL, np.int64)).astype(np.float64)
    Gd, Hd = np.float64(G), np.float64(H)
    left = (gl * gl) / (hl + lam)
    right = (gr * gr) / (hr + lam)
    par = (Gd * Gd) / (Hd + lam)
    return 0.5 * ((left + right) - par)


def _ulps(a, b):
    return int(np.float64(b).view(np.int64)) - int(np.float64(a).view(np.int64))


def _pick(G, H, GL, lam, d, start):
    """Two distinct hessians (HLa, HLb) from start on, for the same GL, with gain(b) exactly d ulps above
    gain(a) (below when d < 0)."""
    HL = start + np.arange(4000, dtype=np.int64)
    bits = _gains(np.full(HL.shape, GL, np.int64), HL, G, H, lam).view(np.int64)
    for i in range(len(HL)):
        j = np.flatnonzero(bits[i + 1:] - bits[i] == d)
        if j.size:
            return int(HL[i]), int(HL[i + 1 + j[0]])
        j = np.flatnonzero(bits[i] - bits[i + 1:] == d)
        if j.size:
            return int(HL[i + 1 + j[0]]), int(HL[i])
    raise AssertionError("no candidate pair found")


def _gain_min(G, H, GL, lam):
    """The hessian HL at which the gain is smallest over HL (the gain is convex in HL: a sum of x^2 / y
    terms)."""
    f = lambda h: float(_gains(np.array([GL]), np.array([h]), G, H, lam)[0])  # noqa: E731
    lo, hi = 1, H - 1
    while hi - lo > 3:
        m1, m2 = lo + (hi - lo) // 3, hi - (hi - lo) // 3
        if f(m1) < f(m2):
            hi = m2
        else:
            lo = m1
    return lo


def _flat_start(G, H, GL, lam):
    """A hessian HL on the rising side of the gain's minimum over HL where one unit of HL moves the gain by
    about a quarter ulp, so that nearby candidates differ by a few ulps."""
    lo = _gain_min(G, H, GL, lam)
    delta = 1 << 16
    while True:
        b = _gains(np.full(2, GL, np.int64), np.array([lo + delta, lo + delta + 4096], np.int64), G, H,
                   lam).view(np.int64)
        if b[1] - b[0] >= 1024:
            return lo + delta
        delta *= 2


class Case:
    def __init__(self, n_nodes, F, n_bins, G, H):
        self.B = n_bins + 1
        self.n_bins, self.G, self.H = n_bins, G, H
        self.h = np.zeros((n_nodes, F, self.B, 2), np.int64)
        for n in range(n_nodes):
            for f in range(F):
                self.weak(n, f)
        self.expect = {}

    def strip(self, n, f, cuts, miss=(0, 0)):
        """cuts: [(t, GL, HL)] ascending in t and HL: the prefix at t is (GL, HL); the rest after the last cut."""
        c = self.h[n, f]
        c[:] = 0
        pg = ph = 0
        for t, gl, hl in cuts:
            c[t] = (gl - pg, hl - ph)
            pg, ph = gl, hl
        c[cuts[-1][0] + 1] = (self.G - pg - miss[0], self.H - ph - miss[1])
        c[self.n_bins] = miss

    def weak(self, n, f):
        """A strip whose every candidate gain is close to 0 (left and right have equal ratios)."""
        self.strip(n, f, [(5 + f % 7, self.G // 2, self.H // 2)])


def _build(n_bins, G, H, GL, lam):
    if H < (1 << 31):
        return _build_near_min(n_bins, G, H, GL, lam)
    F = 24
    c = Case(6, F, n_bins, G, H)
    h0 = _flat_start(G, H, GL, lam)
    t0 = min(40, n_bins - 3)
    # (a) features 3 and 13 (different CTAs of gbt_find_splits and of the level finish): node 0, the later
    # feature higher by 1 ulp; node 1, the earlier one higher by 2 ulps; node 2, an exact tie
    for n, d, win in ((0, 1, 13), (1, -2, 3), (2, 0, 3)):
        ha, hb = _pick(G, H, GL, lam, d, h0 + 97 * n)
        c.strip(n, 3, [(t0, GL, ha)])
        c.strip(n, 13, [(t0 + 1, GL, hb)])
        c.expect[n] = (win, t0 if win == 3 else t0 + 1, 0)
    # (b) four features of one CTA (16..19) with gains x, x+1, x+3, x+2 ulps
    ha, hb1 = _pick(G, H, GL, lam, 1, h0 + 500)
    _, hb3 = _pick(G, H, GL, lam, 3, ha)
    _, hb2 = _pick(G, H, GL, lam, 2, ha)
    for f, hl in zip((16, 17, 18, 19), (ha, hb1, hb3, hb2)):
        c.strip(3, f, [(t0 + f - 16, GL, hl)])
    c.expect[3] = (18, t0 + 2, 0)
    # (c) two cuts of feature 21 without missing mass, the later one higher by 2 ulps
    ha, hb = _pick(G, H, GL, lam, 2, h0 + 900)
    c.strip(4, 21, [(t0, GL, ha), (t0 + 3, GL, hb)])
    c.expect[4] = (21, t0 + 3, 0)
    # (d) one cut of feature 9 whose missing rows (G 0, H m) make missing-left 1 ulp higher than missing-right
    ha, hb = _pick(G, H, GL, lam, 1, h0 + 1300)
    c.strip(5, 9, [(t0, GL, ha)], miss=(0, hb - ha))
    c.expect[5] = (9, t0, 1)
    return c


def _build_near_min(n_bins, G, H, GL, lam):
    """The cases of _build for sums below 2^31, where every partial sum of a strip fits in 32 bits. One unit
    of HL then moves the gain by many ulps except near its minimum over HL, where the gain is flat to within
    its rounding: every pair comes from a window of hessians around the minimum, each partner found for the
    given first hessian."""
    F = 24
    c = Case(6, F, n_bins, G, H)
    m = _gain_min(G, H, GL, lam)
    HL = np.arange(m - 3000, m + 3000, dtype=np.int64)
    bits = _gains(np.full(HL.shape, GL, np.int64), HL, G, H, lam).view(np.int64)

    def partner(i, d, above=False):
        """An index j (j > i when above) whose gain is exactly d ulps above gain i, or None."""
        j = np.flatnonzero(bits - bits[i] == d)
        j = j[(j > i) if above else (j != i)]
        return int(j[0]) if j.size else None

    def first(ds, above=False, start=0):
        for i in range(start, len(HL)):
            js = [partner(i, d, above) for d in ds]
            if all(j is not None for j in js):
                return [int(HL[i])] + [int(HL[j]) for j in js]
        raise AssertionError("no candidate set found")

    t0 = min(40, n_bins - 3)
    for n, d, win in ((0, 1, 13), (1, -2, 3), (2, 0, 3)):
        ha, hb = first([d], start=97 * n)
        c.strip(n, 3, [(t0, GL, ha)])
        c.strip(n, 13, [(t0 + 1, GL, hb)])
        c.expect[n] = (win, t0 if win == 3 else t0 + 1, 0)
    ha, hb1, hb3, hb2 = first([1, 3, 2], start=500)
    for f, hl in zip((16, 17, 18, 19), (ha, hb1, hb3, hb2)):
        c.strip(3, f, [(t0 + f - 16, GL, hl)])
    c.expect[3] = (18, t0 + 2, 0)
    ha, hb = first([2], above=True, start=900)
    c.strip(4, 21, [(t0, GL, ha), (t0 + 3, GL, hb)])
    c.expect[4] = (21, t0 + 3, 0)
    ha, hb = first([1], above=True, start=1300)
    c.strip(5, 9, [(t0, GL, ha)], miss=(0, hb - ha))
    c.expect[5] = (9, t0, 1)
    return c


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g
    from histogram_construction_gb300.session import Session, splits_to_numpy
    g.lib()
    return g, Session, splits_to_numpy


def _session(Session, n_bins, F):
    s = Session()
    wide = n_bins > 255
    s.upload_bins(np.zeros((F, 8), np.uint16 if wide else np.uint8), n_bins, 0xFFFF if wide else 0xFF)
    s.begin_tree(np.zeros((8, 2), np.float32), 1.0, 1.0)
    return s


def _same(got, ref, where):
    for k in ("feature", "bin", "default_left", "g_left", "h_left", "g_right", "h_right"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{where} field {k}")
    np.testing.assert_array_equal(got["gain"].view(np.int64), ref["gain"].view(np.int64), err_msg=f"{where} gain")


def _check_designed(case, ref, where):
    for n, (f, t, dl) in case.expect.items():
        assert (int(ref["feature"][n]), int(ref["bin"][n]), int(ref["default_left"][n])) == (f, t, dl), (where, n)


SETTINGS = [
    # (n_bins, G, H, GL, lambda): staged u8 strips / strips in global memory; fast screen (sums below 2^45),
    # checked screen (sums beyond 2^45), no screen (lambda < 0)
    (255, 3 << 36, 1 << 44, 5 << 40, 1.0),
    (255, 3 << 40, 1 << 47, 5 << 44, 0.5),
    (255, 3 << 36, 1 << 44, 5 << 40, -0.25),
    (4096, 3 << 36, 1 << 44, 5 << 40, 1.0),
    (4096, 3 << 40, 1 << 47, 5 << 44, 0.5),
    (4096, 3 << 36, 1 << 44, 5 << 40, -0.25),
    # sums below 2^31 (the scan's 32-bit instantiation), staged and in global memory
    (255, 3 << 26, 1 << 30, 5 << 26, 1.0),
    (255, 3 << 26, 1 << 30, 5 << 26, 0.5),
    (4096, 3 << 26, 1 << 30, 5 << 26, 1.0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("n_bins,G,H,GL,lam", SETTINGS)
def test_find_splits_near_ties(gb, oracle_mod, n_bins, G, H, GL, lam):
    g, Session, s2n = gb
    case = _build(n_bins, G, H, GL, lam)
    ref, st = oracle_mod.find_splits(case.h, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
    assert st == oracle_mod.OK
    _check_designed(case, ref, "oracle")
    s = _session(Session, n_bins, case.h.shape[1])
    try:
        got = s2n(s.find_splits(torch.from_numpy(case.h).cuda(), lam=lam))
        assert s.sync() == 0
    finally:
        s.close()
    _same(got, ref, f"find n_bins={n_bins} lam={lam}")


@pytest.mark.gpu
@pytest.mark.parametrize("n_bins,G,H,GL,lam", SETTINGS)
def test_level_finish_near_ties(gb, oracle_mod, n_bins, G, H, GL, lam):
    """The fused subtraction + split find of both siblings: the small histograms carry the near ties, and
    so do the large ones (the same cases with the node order reversed), parent = small + large."""
    g, Session, s2n = gb
    case = _build(n_bins, G, H, GL, lam)
    small = case.h
    large = case.h[::-1].copy()
    parent = small + large
    ref_s, _ = oracle_mod.find_splits(small, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
    ref_l, _ = oracle_mod.find_splits(large, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
    ref_large, st = oracle_mod.subtract(parent, None, small)
    assert st == oracle_mod.OK and np.array_equal(ref_large, large)
    s = _session(Session, n_bins, small.shape[1])
    try:
        got_large, so, lo = s.subtract_and_find(torch.from_numpy(parent).cuda(), torch.from_numpy(small).cuda(),
                                                lam=lam)
        assert s.sync() == 0
        np.testing.assert_array_equal(got_large.cpu().numpy(), large)
        _same(s2n(so), ref_s, f"finish small n_bins={n_bins} lam={lam}")
        _same(s2n(lo), ref_l, f"finish large n_bins={n_bins} lam={lam}")
    finally:
        s.close()


def _widened(case, n_features=700, moves=((13, 301), (9, 450), (17, 602))):
    """The case's histograms with features appended (copies of features 0-2, weak in every node) up to
    n_features, and some designed features moved far away (swapped with appended ones), so that the
    near-tied candidates fall in different CTAs and in different passes of one CTA of a grid of many
    waves."""
    h = case.h
    extra = np.tile(h[:, 0:3], (1, (n_features - h.shape[1] + 2) // 3, 1, 1))[:, : n_features - h.shape[1]]
    h = np.concatenate([h, extra], axis=1)
    for a, b in moves:
        h[:, [a, b]] = h[:, [b, a]]
    return np.ascontiguousarray(h)


@pytest.mark.gpu
@pytest.mark.parametrize("n_bins,G,H,GL,lam", [x for x in SETTINGS if x[0] == 255])
def test_level_finish_near_ties_many_waves(gb, oracle_mod, n_bins, G, H, GL, lam):
    """test_level_finish_near_ties on 700 features: the fused finish runs its many-wave form (several
    groups of four features per CTA, in passes)."""
    g, Session, s2n = gb
    small = _widened(_build(n_bins, G, H, GL, lam))
    large = small[::-1].copy()
    parent = small + large
    ref_s, _ = oracle_mod.find_splits(small, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
    ref_l, _ = oracle_mod.find_splits(large, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
    assert set(int(x) for x in ref_s["feature"]) <= {3, 301, 450, 16, 602, 18, 19, 21}
    s = _session(Session, n_bins, small.shape[1])
    try:
        got_large, so, lo = s.subtract_and_find(torch.from_numpy(parent).cuda(), torch.from_numpy(small).cuda(),
                                                lam=lam)
        assert s.sync() == 0
        np.testing.assert_array_equal(got_large.cpu().numpy(), large)
        _same(s2n(so), ref_s, f"finish small many waves lam={lam}")
        _same(s2n(lo), ref_l, f"finish large many waves lam={lam}")
    finally:
        s.close()


def test_near_tie_cases_are_what_they_claim(oracle_mod):
    """CPU check of the case builder against the oracle's gain: each designed pair differs by the stated
    number of ulps (runs without a GPU)."""
    for n_bins, G, H, GL, lam in SETTINGS[:3]:
        for d in (0, 1, 2, 3, 4, -2):
            ha, hb = _pick(G, H, GL, lam, d, _flat_start(G, H, GL, lam))
            ga = oracle_mod.gain(float(GL), float(ha), float(G - GL), float(H - ha), float(G), float(H), lam, 0.0)
            gb_ = oracle_mod.gain(float(GL), float(hb), float(G - GL), float(H - hb), float(G), float(H), lam, 0.0)
            assert _ulps(ga, gb_) == d and ha != hb
        case = _build(n_bins, G, H, GL, lam)
        assert (case.h[..., 1] >= 0).all()
        ref, st = oracle_mod.find_splits(case.h, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
        assert st == oracle_mod.OK
        _check_designed(case, ref, "oracle")
    for n_bins, G, H, GL, lam in SETTINGS[6:]:
        case = _build(n_bins, G, H, GL, lam)
        assert (case.h[..., 1] >= 0).all()
        assert np.abs(case.h[..., 0]).sum(axis=2).max() < 2 ** 31 and case.h[..., 1].sum(axis=2).max() < 2 ** 31
        ref, st = oracle_mod.find_splits(case.h, n_bins, lam, 0.0, 0.0, 1.0, 1.0)
        assert st == oracle_mod.OK
        _check_designed(case, ref, "oracle")


def _empty_first_cut_case(n_bins):
    """One node, one feature: slot 0 empty, 100 real slots of (G -1, H 1), missing (G 100, H 10). Sending only
    the missing rows left (cut 0, missing left) ties exactly with cut n_bins - 1, missing right (the same two
    sides swapped); the serial order picks cut 0."""
    B = n_bins + 1
    h = np.zeros((1, 1, B, 2), np.int64)
    h[0, 0, 1:101] = (-1, 1)
    h[0, 0, n_bins] = (100, 10)
    return h


def test_empty_first_cut_oracle_pin(oracle_mod):
    for n_bins in (255, 4096):
        ref, st = oracle_mod.find_splits(_empty_first_cut_case(n_bins), n_bins, 1.0, 0.0, 0.0, 1.0, 1.0)
        assert st == oracle_mod.OK
        assert (int(ref["feature"][0]), int(ref["bin"][0]), int(ref["default_left"][0])) == (0, 0, 1)
        expect = 0.5 * ((100.0 * 100.0 / 11.0 + 100.0 * 100.0 / 101.0) - 0.0)
        assert ref["gain"][0] == expect


@pytest.mark.gpu
@pytest.mark.parametrize("n_bins", [255, 4096])
def test_empty_first_cut_on_gpu(gb, oracle_mod, n_bins):
    """Cuts over empty cells repeat the previous cut and are skipped by the scan, except cut 0."""
    g, Session, s2n = gb
    h = _empty_first_cut_case(n_bins)
    ref, _ = oracle_mod.find_splits(h, n_bins, 1.0, 0.0, 0.0, 1.0, 1.0)
    s = _session(Session, n_bins, 1)
    try:
        got = s2n(s.find_splits(torch.from_numpy(h).cuda()))
        parent = np.concatenate([h, h]).sum(axis=0, keepdims=True)
        large, so, lo = s.subtract_and_find(torch.from_numpy(parent).cuda(), torch.from_numpy(h).cuda())
        assert s.sync() == 0
    finally:
        s.close()
    _same(got, ref, "find")
    _same(s2n(so), ref, "finish small")
    _same(s2n(lo), ref, "finish large")
