"""GPU parity of the multi-output (vector-leaf) histogram build against the serial oracle.

Bar: int64 cells bit-exact for every target; each target's histogram equals the
one-target build of that target's pairs.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g
    from histogram_construction_gb300.session import Session
    g.lib()
    return g, Session


@pytest.fixture(scope="module")
def oracle():
    import oracle as o
    return o


def _scales(g, gp):
    sg, sh = [], []
    for t in range(gp.shape[1]):
        s, a, b = g.gbt_suggest_scales(0, float(np.abs(gp[:, t, 0]).max()), float(np.abs(gp[:, t, 1]).max()))
        assert s == 0
        sg.append(a)
        sh.append(b)
    return sg, sh


def _check_level(sess, oracle, w, q, rows, offs, where):
    h = sess.build_level_multi(rows, offs)
    assert sess.sync() == 0
    offs_h = offs.cpu().numpy() if torch.is_tensor(offs) else offs
    rows_h = rows.cpu().numpy() if torch.is_tensor(rows) else rows
    ref, st = oracle.build_hist_multi(w.bins, w.n_bins, w.sentinel, q, rows_h, offs_h)
    assert st == oracle.OK
    np.testing.assert_array_equal(h.cpu().numpy(), ref, err_msg=where)
    return h


@pytest.mark.parametrize("k", [1, 2, 3, 4, 5, 8])
def test_level5_reduced_all_target_counts(gb, oracle, k):
    """37 features: two feature tiles, the second ragged (5 of 16 in its first quarter); targets in groups of
    four, the last group partial for k = 5."""
    g, Session = gb
    w = synth.make("level5", n_rows=90_000, n_features=37, depth=3)
    gp = synth.gpair_multi("level5", w.n_rows, k)
    sg, sh = _scales(g, gp)
    q, st = oracle.quantise_multi(gp, sg, sh)
    assert st == oracle.OK
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        s.begin_tree_multi(torch.from_numpy(gp).cuda(), sg, sh)
        for d in (2, 3):
            lv = w.levels[d]
            _check_level(s, oracle, w, q, lv.built_rows, lv.built_offsets, f"k={k} depth {d} built")
        _check_level(s, oracle, w, q, w.levels[2].rows, torch.from_numpy(w.levels[2].offsets).cuda(),
                     f"k={k} depth 2 all")


def test_each_target_equals_the_single_build(gb, oracle):
    g, Session = gb
    w = synth.make("level5", n_rows=60_000, n_features=70, depth=2)
    k = 3
    gp = synth.gpair_multi("level5", w.n_rows, k)
    sg, sh = _scales(g, gp)
    lv = w.levels[2]
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        s.begin_tree_multi(gp, sg, sh)  # host gpair
        hm = s.build_level_multi(lv.rows, lv.offsets)
        assert s.sync() == 0
        hm = hm.cpu().numpy()
        for t in range(k):
            s.begin_tree(np.ascontiguousarray(gp[:, t, :]), sg[t], sh[t])
            h1 = s.build_level(lv.rows, lv.offsets)
            assert s.sync() == 0
            np.testing.assert_array_equal(hm[t], h1.cpu().numpy(), err_msg=f"target {t}")


def test_root_identity_rows_and_empty_nodes(gb, oracle):
    g, Session = gb
    w = synth.make("root")
    k = 4
    gp = synth.gpair_multi("root", w.n_rows, k)
    sg, sh = _scales(g, gp)
    q, _ = oracle.quantise_multi(gp, sg, sh)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        s.begin_tree_multi(gp, sg, sh)
        _check_level(s, oracle, w, q, None, np.array([0, w.n_rows], np.int64), "root")
        rows = np.arange(w.n_rows, dtype=np.int32)[::-1].copy()
        offs = np.array([0, 0, 1, 1, 5000, w.n_rows, w.n_rows], np.int64)  # empty and 1-row nodes
        _check_level(s, oracle, w, q, rows, offs, "edge nodes")


def test_unsupported_and_errors(gb, oracle):
    g, Session = gb
    w = synth.make("u16miss", n_rows=5000, n_features=4, depth=1)
    gp = synth.gpair_multi("u16miss", w.n_rows, 2)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        s.begin_tree_multi(gp, [1024.0, 1024.0], [1024.0, 1024.0])
        hist = torch.empty((2, 1, 4, w.n_bins + 1, 2), dtype=torch.int64, device="cuda")
        offs = torch.tensor([0, w.n_rows], dtype=torch.int64, device="cuda")
        st = g.gbt_build_level_multi(s.ctx, None, offs, 1, hist)
        assert st == g.GBT_ERR_UNSUPPORTED
        assert g.gbt_begin_tree_multi(s.ctx, gp, 17, [1.0] * 17, [1.0] * 17) == g.GBT_ERR_UNSUPPORTED
        assert g.gbt_begin_tree_multi(s.ctx, gp, 2, [1.0, 0.0], [1.0, 1.0]) == g.GBT_ERR_INVALID_ARG
    w = synth.make("root")
    gp = synth.gpair_multi("root", w.n_rows, 2)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel)
        # a scale that sends |q| past 2^21 - 1: the overflow is reported at sync
        assert g.gbt_begin_tree_multi(s.ctx, gp, 2, [1.0, 1e7], [1.0, 1.0]) == g.GBT_OK
        assert s.sync() == g.GBT_ERR_QUANT_OVERFLOW


def test_level5_full_size_three_targets(gb, oracle):
    """The full 1M x 100 depth-5 level, three targets (the pages' multi-output benchmark has three)."""
    g, Session = gb
    w = synth.make("level5")
    k = 3
    gp = synth.gpair_multi("level5", w.n_rows, k)
    sg, sh = _scales(g, gp)
    q, _ = oracle.quantise_multi(gp, sg, sh)
    lv = w.levels[5]
    with Session() as s:
        s.upload_bins(torch.from_numpy(w.bins).cuda(), w.n_bins, w.sentinel)
        s.begin_tree_multi(torch.from_numpy(gp).cuda(), sg, sh)
        _check_level(s, oracle, w, q, lv.built_rows, lv.built_offsets, "level5 full k=3")
