"""GPU parity: the CUDA path through the C ABI against the serial CPU oracle.

Bar: int64 histograms bit-exact; split (feature, bin, default_left, sums)
bit-exact; gains compared bit-for-bit as doubles (the kernels evaluate the
same IEEE operations in the same order with no contraction; the stated
tolerance for gains is 1e-5 relative, which exact equality implies).
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
    from histogram_construction_gb300.session import Session, splits_to_numpy
    g.lib()
    return g, Session, splits_to_numpy


def _scales(w):
    import histogram_construction_gb300 as g
    mg = float(np.abs(w.gpair[:, 0]).max())
    mh = float(np.abs(w.gpair[:, 1]).max())
    s, sg, sh = g.gbt_suggest_scales(0, mg, mh)
    assert s == 0
    return sg, sh


def assert_splits_equal(gpu, ref, where=""):
    assert gpu.shape == ref.shape, where
    for k in ("feature", "bin", "default_left", "g_left", "h_left", "g_right", "h_right"):
        np.testing.assert_array_equal(gpu[k], ref[k], err_msg=f"{where} field {k}")
    # gains bit-for-bit (covers -inf for nodes without a valid split)
    np.testing.assert_array_equal(gpu["gain"].view(np.int64), ref["gain"].view(np.int64), err_msg=f"{where} gain")


def run_level(sess, oracle, w, depth, sg, sh, lam=1.0, gamma=0.0, mcw=0.0, host_offsets=False):
    """Build parents (depth-1, all rows) and the smaller siblings at depth, then subtract+find.
    Compares every histogram and split with the oracle."""
    q, st = oracle.quantise(w.gpair, sg, sh)
    assert st == oracle.OK
    par, lv = w.levels[depth - 1], w.levels[depth]
    # parents
    offs_p = par.offsets if host_offsets else torch.from_numpy(par.offsets).cuda()
    hp = sess.build_level(par.rows, offs_p)
    ref_hp, st = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, par.rows, par.offsets)
    assert st == oracle.OK
    # smaller siblings
    offs_s = lv.built_offsets if host_offsets else torch.from_numpy(lv.built_offsets).cuda()
    hs = sess.build_level(lv.built_rows, offs_s)
    ref_hs, st = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, lv.built_rows, lv.built_offsets)
    large, so, lo = sess.subtract_and_find(hp, hs, lam=lam, gamma=gamma, mcw=mcw)
    assert sess.sync() == 0, sess
    np.testing.assert_array_equal(hp.cpu().numpy(), ref_hp, err_msg="parent hist")
    np.testing.assert_array_equal(hs.cpu().numpy(), ref_hs, err_msg="small hist")
    ref_large, st = oracle.subtract(ref_hp, None, ref_hs)
    assert st == oracle.OK
    np.testing.assert_array_equal(large.cpu().numpy(), ref_large, err_msg="large hist")
    ref_so, _ = oracle.find_splits(ref_hs, w.n_bins, lam, gamma, mcw, sg, sh)
    ref_lo, _ = oracle.find_splits(ref_large, w.n_bins, lam, gamma, mcw, sg, sh)
    from histogram_construction_gb300.session import splits_to_numpy
    assert_splits_equal(splits_to_numpy(so), ref_so, "small splits")
    assert_splits_equal(splits_to_numpy(lo), ref_lo, "large splits")
    # the fused level step (build partials -> subtract -> find in one pass) gives the same bytes
    hs2, large2, so2, lo2 = sess.level_step(lv.built_rows, offs_s, hp, lam=lam, gamma=gamma, mcw=mcw)
    assert sess.sync() == 0
    np.testing.assert_array_equal(hs2.cpu().numpy(), ref_hs, err_msg="level_step small hist")
    np.testing.assert_array_equal(large2.cpu().numpy(), ref_large, err_msg="level_step large hist")
    assert_splits_equal(splits_to_numpy(so2), ref_so, "level_step small splits")
    assert_splits_equal(splits_to_numpy(lo2), ref_lo, "level_step large splits")
    return hp, hs, large, ref_hp, ref_hs, ref_large


# --------------------------------------------------------------------------- workloads at parity-test size
def test_root_full_size(gb, oracle_mod):
    g, Session, s2n = gb
    w = synth.make("root")
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        lv = w.levels[0]
        h = s.build_level(None, lv.offsets)
        out = s.find_splits(h, lam=1.0)
        assert s.sync() == 0
        q, _ = oracle_mod.quantise(w.gpair, sg, sh)
        ref, st = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, None, lv.offsets)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        rs, _ = oracle_mod.find_splits(ref, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
        assert_splits_equal(s2n(out), rs, "root")


@pytest.mark.parametrize("n_rows", [30_000, 60_000])
def test_level_step_pinned_host_buffers(gb, oracle_mod, n_rows):
    """gbt_level_step with page-locked host buffers: the row list, the offsets and the split records are
    read and written in place by the kernels (pageable host buffers, copied first, are the other tests')."""
    g, Session, s2n = gb
    w = synth.make("level5", n_rows=n_rows)
    sg, sh = _scales(w)
    q, _ = oracle_mod.quantise(w.gpair, sg, sh)
    par, lv = w.levels[4], w.levels[5]
    ref_hp, _ = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, par.rows, par.offsets)
    ref_hs, _ = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, lv.built_rows, lv.built_offsets)
    ref_large, _ = oracle_mod.subtract(ref_hp, None, ref_hs)
    ref_so, _ = oracle_mod.find_splits(ref_hs, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
    ref_lo, _ = oracle_mod.find_splits(ref_large, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        hp = s.build_level(par.rows, torch.from_numpy(par.offsets).cuda())
        n_p = len(lv.built_offsets) - 1
        rows_h = torch.from_numpy(lv.built_rows).pin_memory()
        offs_h = torch.from_numpy(lv.built_offsets).pin_memory()
        so_h = torch.zeros((n_p, g.SPLIT_BYTES), dtype=torch.uint8).pin_memory()
        lo_h = torch.zeros((n_p, g.SPLIT_BYTES), dtype=torch.uint8).pin_memory()
        hs = s.hist_tensor(n_p)
        large = torch.empty_like(hs)
        s.check(g.gbt_level_step(s.ctx, rows_h, offs_h, n_p, hp, None, hs, large, g.params(1.0, 0.0, 0.0), so_h,
                                 lo_h))
        assert s.sync() == 0
        np.testing.assert_array_equal(hs.cpu().numpy(), ref_hs, err_msg="small hist")
        np.testing.assert_array_equal(large.cpu().numpy(), ref_large, err_msg="large hist")
        assert_splits_equal(s2n(so_h), ref_so, "pinned small splits")
        assert_splits_equal(s2n(lo_h), ref_lo, "pinned large splits")


@pytest.mark.parametrize("plan_kernel", [False, True])
@pytest.mark.parametrize("n_rows,host_offsets", [(60_000, False), (200_000, True)])
def test_level5_reduced(gb, oracle_mod, monkeypatch, n_rows, host_offsets, plan_kernel):
    """plan_kernel: the level planned by the plan kernel instead of by the histogram kernel itself."""
    g, Session, s2n = gb
    if plan_kernel:
        monkeypatch.setenv("GBT_PLAN_KERNEL", "1")
    w = synth.make("level5", n_rows=n_rows)
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        run_level(s, oracle_mod, w, 5, sg, sh, host_offsets=host_offsets)


def test_level5_full_size(gb, oracle_mod):
    """1,000,000 x 100 u8, level 5: the benchmark's own launch configuration, compared in full."""
    g, Session, s2n = gb
    w = synth.make("level5")
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(torch.from_numpy(w.bins).cuda(), w.n_bins, w.sentinel)
        s.begin_tree(torch.from_numpy(w.gpair).cuda(), sg, sh)
        run_level(s, oracle_mod, w, 5, sg, sh)


def test_wide_reduced(gb, oracle_mod):
    g, Session, s2n = gb
    w = synth.make("wide", n_rows=8192, n_features=4133)  # ragged last tile (37 of 64 features)
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        run_level(s, oracle_mod, w, 3, sg, sh, lam=0.5, gamma=0.1)


def test_wide_full_size(gb, oracle_mod):
    """131,072 x 16,384 u8, level 3: the 4 parents (all rows), the 4 smaller siblings and their
    splits, compared in full (the oracle builds every histogram itself)."""
    g, Session, s2n = gb
    w = synth.make("wide")
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(torch.from_numpy(w.bins).cuda(), w.n_bins, w.sentinel)
        s.begin_tree(torch.from_numpy(w.gpair).cuda(), sg, sh)
        run_level(s, oracle_mod, w, 3, sg, sh)


@pytest.mark.parametrize("plan_kernel", [False, True])
def test_u16_missing_reduced(gb, oracle_mod, monkeypatch, plan_kernel):
    g, Session, s2n = gb
    if plan_kernel:
        monkeypatch.setenv("GBT_PLAN_KERNEL", "1")
    w = synth.make("u16miss", n_rows=100_000, n_features=20, depth=5)
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        run_level(s, oracle_mod, w, 5, sg, sh, mcw=0.5)


def test_u16_missing_full_size(gb, oracle_mod):
    """2,000,000 x 64 u16 (40% missing), level 7: 64 built + 64 derived nodes, compared in full."""
    g, Session, s2n = gb
    w = synth.make("u16miss")
    sg, sh = _scales(w)
    with Session() as s:
        s.upload_bins(torch.from_numpy(w.bins).cuda(), w.n_bins, w.sentinel)
        s.begin_tree(torch.from_numpy(w.gpair).cuda(), sg, sh)
        run_level(s, oracle_mod, w, 7, sg, sh)


def test_dense_tree_with_device_partition(gb, oracle_mod):
    """Dense u8 with constant h: levels 0..4 of a real tree. Each level's splits come from the device,
    the device partition routes the rows by them, and the oracle follows the same steps."""
    g, Session, s2n = gb
    w = synth.make("dense", n_rows=120_000, n_features=130, depth=1)
    sg, sh = _scales(w)
    q, _ = oracle_mod.quantise(w.gpair, sg, sh)
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        offs = np.array([0, w.n_rows], np.int64)
        h = s.build_level(None, offs)
        sp = s.find_splits(h)
        ref_h, _ = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, None, offs)
        assert s.sync() == 0
        np.testing.assert_array_equal(h.cpu().numpy(), ref_h)
        ref_sp, _ = oracle_mod.find_splits(ref_h, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
        assert_splits_equal(s2n(sp), ref_sp, "level 0")
        d_rows, ref_rows = None, None
        for depth in range(1, 5):
            d_rows, d_offs = s.partition(d_rows, offs, sp)
            ref_rows, ref_offs, st = oracle_mod.partition(w.bins, w.n_bins, w.sentinel, ref_rows, offs, ref_sp)
            assert st == oracle_mod.OK and s.sync() == 0
            np.testing.assert_array_equal(d_rows.cpu().numpy(), ref_rows, err_msg=f"rows depth {depth}")
            np.testing.assert_array_equal(d_offs.cpu().numpy(), ref_offs, err_msg=f"offsets depth {depth}")
            offs = ref_offs
            n_nodes = len(offs) - 1
            sizes = np.diff(offs)
            small = np.where(sizes[1::2] < sizes[0::2], np.arange(1, n_nodes, 2), np.arange(0, n_nodes, 2))
            large_ids = small ^ 1
            b_rows = np.concatenate([ref_rows[offs[i]:offs[i + 1]] for i in small]).astype(np.int32)
            b_offs = np.concatenate([[0], np.cumsum(sizes[small])]).astype(np.int64)
            hs = s.build_level(b_rows, b_offs)
            large, so, lo = s.subtract_and_find(h, hs)
            ref_hs, _ = oracle_mod.build_hist(w.bins, w.n_bins, w.sentinel, q, b_rows, b_offs)
            ref_large, _ = oracle_mod.subtract(ref_h, None, ref_hs)
            assert s.sync() == 0
            np.testing.assert_array_equal(hs.cpu().numpy(), ref_hs, err_msg=f"small depth {depth}")
            np.testing.assert_array_equal(large.cpu().numpy(), ref_large, err_msg=f"large depth {depth}")
            ref_h = np.empty((n_nodes,) + ref_hs.shape[1:], np.int64)
            ref_h[small] = ref_hs
            ref_h[large_ids] = ref_large
            ref_sp, _ = oracle_mod.find_splits(ref_h, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
            gpu_sp = np.empty(n_nodes, dtype=ref_sp.dtype)
            gpu_sp[small] = s2n(so)
            gpu_sp[large_ids] = s2n(lo)
            assert_splits_equal(gpu_sp, ref_sp, f"depth {depth}")
            h = hs.new_empty((n_nodes,) + tuple(hs.shape[1:]))
            h[torch.from_numpy(small).cuda()] = hs
            h[torch.from_numpy(large_ids).cuda()] = large
            sp = torch.from_numpy(gpu_sp.view(np.uint8).reshape(n_nodes, -1).copy()).cuda()


# --------------------------------------------------------------------------- edge cases
def _tiny(width=1, n_rows=300, n_features=5, n_bins=12, miss=0.2, seed=0):
    rng = np.random.default_rng(seed)
    sentinel = 0xFF if width == 1 else 0xFFFF
    dt = np.uint8 if width == 1 else np.uint16
    bins = rng.integers(0, n_bins, size=(n_features, n_rows)).astype(dt)
    bins[rng.random(bins.shape) < miss] = sentinel
    gp = np.stack([rng.standard_normal(n_rows), rng.uniform(0.1, 1, n_rows)], 1).astype(np.float32)
    return bins, gp, sentinel


@pytest.mark.parametrize("width", [1, 2])
def test_edge_nodes_empty_single_unsorted(gb, oracle_mod, width):
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(width, n_rows=5000, n_features=70 if width == 1 else 33, n_bins=63)
    rng = np.random.default_rng(3)
    perm = rng.permutation(5000).astype(np.int32)  # unsorted rows inside nodes
    rows = perm[:4000]
    offs = np.array([0, 0, 1, 1, 2500, 2500, 4000], np.int64)  # empty, 1-row, empty, big, empty, rest
    with Session() as s:
        s.upload_bins(bins, 63, sentinel).begin_tree(gp, 1024.0, 1000.0)
        h = s.build_level(rows, offs)
        sp = s.find_splits(h, lam=1.0, mcw=0.1)
        assert s.sync() == 0
        q, _ = oracle_mod.quantise(gp, 1024.0, 1000.0)
        ref, _ = oracle_mod.build_hist(bins, 63, sentinel, q, rows, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        rs, _ = oracle_mod.find_splits(ref, 63, 1.0, 0.0, 0.1, 1024.0, 1000.0)
        assert_splits_equal(s2n(sp), rs)


@pytest.mark.parametrize("width", [1, 2])
@pytest.mark.parametrize("target_items", [None, "7", "1000"])
def test_many_nodes_and_item_targets(gb, oracle_mod, monkeypatch, width, target_items):
    """700 nodes (three planning batches of 256), with empty and one-row nodes: the level's histograms,
    splits and the fused level step. target_items overrides the plan's item target: 7 gives far fewer
    chunks wanted than nodes, 1000 several items per CTA taken from the counter."""
    g, Session, s2n = gb
    if target_items is not None:
        monkeypatch.setenv("GBT_TARGET_ITEMS", target_items)
    n_rows = 60_000
    bins, gp, sentinel = _tiny(width, n_rows=n_rows, n_features=70 if width == 1 else 20, n_bins=50, seed=11)
    rng = np.random.default_rng(12)
    sizes = rng.integers(0, 140, size=700)
    sizes[::37] = 0
    sizes[5::41] = 1
    sizes[9] = 4000  # one node larger than a chunk
    assert sizes.sum() <= n_rows
    rows = rng.permutation(n_rows)[: int(sizes.sum())].astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
    sg, sh = 1024.0, 1000.0
    q, _ = oracle_mod.quantise(gp, sg, sh)
    with Session() as s:
        s.upload_bins(bins, 50, sentinel).begin_tree(gp, sg, sh)
        h = s.build_level(rows, offs)
        sp = s.find_splits(h, lam=1.0)
        assert s.sync() == 0
        ref, st = oracle_mod.build_hist(bins, 50, sentinel, q, rows, offs)
        assert st == oracle_mod.OK
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        rs, _ = oracle_mod.find_splits(ref, 50, 1.0, 0.0, 0.0, sg, sh)
        assert_splits_equal(s2n(sp), rs, "700 nodes")
        # pairs (2i, 2i + 1): parents hold both children's rows; child 2i is built, 2i + 1 derived
        hp = s.build_level(rows, offs[::2])
        small_rows = np.concatenate([rows[offs[2 * i]:offs[2 * i + 1]] for i in range(350)])
        small_offs = np.concatenate([[0], np.cumsum(sizes[::2])]).astype(np.int64)
        hs, large, so, lo = s.level_step(small_rows, small_offs, hp, lam=1.0)
        assert s.sync() == 0
        np.testing.assert_array_equal(hs.cpu().numpy(), ref[::2], err_msg="level_step small")
        np.testing.assert_array_equal(large.cpu().numpy(), ref[1::2], err_msg="level_step large")
        assert_splits_equal(s2n(so), rs[::2], "level_step small splits")
        assert_splits_equal(s2n(lo), rs[1::2], "level_step large splits")


def test_edge_all_rows_one_bin_and_all_missing(gb, oracle_mod):
    g, Session, s2n = gb
    N = 20000
    bins = np.full((3, N), 7, np.uint8)
    bins[1] = 0xFF  # feature 1 entirely missing
    gp = np.stack([np.linspace(-1, 1, N), np.full(N, 0.5)], 1).astype(np.float32)
    with Session() as s:
        s.upload_bins(bins, 255, 0xFF).begin_tree(gp, 4096.0, 4096.0)
        offs = np.array([0, N], np.int64)
        h = s.build_level(None, offs)
        sp = s.find_splits(h)
        assert s.sync() == 0
        q, _ = oracle_mod.quantise(gp, 4096.0, 4096.0)
        ref, _ = oracle_mod.build_hist(bins, 255, 0xFF, q, None, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        rs, _ = oracle_mod.find_splits(ref, 255, 1.0, 0.0, 0.0, 4096.0, 4096.0)
        assert_splits_equal(s2n(sp), rs)
        assert rs["feature"][0] == -1


def test_edge_quantisation_limit_forces_minimum_chunks(gb, oracle_mod):
    """|q| at the limit 2^21 - 1: chunks of 1024 rows, nodes built from several chunks."""
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(1, n_rows=5000, n_features=65, n_bins=40)
    gp[:, 0] = np.clip(gp[:, 0], -1.0, 1.0)
    gp[0, 0] = 1.0
    scale = 2097151.0  # q = 2097151 for g = 1.0
    with Session() as s:
        s.upload_bins(bins, 40, sentinel).begin_tree(gp, scale, 1.0e6)
        offs = np.array([0, 3700, 5000], np.int64)
        h = s.build_level(None, offs)
        assert s.sync() == 0
        q, st = oracle_mod.quantise(gp, scale, 1.0e6)
        assert st == oracle_mod.OK and oracle_mod.max_abs_q(q) == 2097151
        ref, _ = oracle_mod.build_hist(bins, 40, sentinel, q, None, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref)
        bad = gp.copy()
        bad[3, 0] = 1.5  # 1.5 * (2^21 - 1): inside the definition's domain, beyond the library's per-row limit
        qb, st = oracle_mod.quantise(bad, scale, 1.0e6)
        assert st == oracle_mod.OK and oracle_mod.max_abs_q(qb) > 2097151
        ref_b, st = oracle_mod.build_hist(bins, 40, sentinel, qb, None, offs)
        assert st == oracle_mod.OK
        assert g.gbt_begin_tree(s.ctx, bad, scale, 1.0e6) == 0
        assert s.sync() == g.GBT_ERR_QUANT_OVERFLOW


@pytest.mark.parametrize("qbig", [2 ** 21, 2 ** 24 + 2, 2 ** 31 - 128])
def test_library_refuses_what_the_oracle_accepts(gb, oracle_mod, qbig):
    """|q| in [2^21, 2^31): the definition's domain, beyond the library's documented per-row limit. The
    oracle builds the histogram; the library reports GBT_ERR_QUANT_OVERFLOW at sync, and its level calls
    then build nothing that could be mistaken for a result."""
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(1, n_rows=3000, n_features=9, n_bins=30)
    gp[:, 0] = np.clip(gp[:, 0], -1.0, 1.0)
    gp[17, 0] = float(qbig)
    q, st = oracle_mod.quantise(gp, 1.0, 1.0e4)
    assert st == oracle_mod.OK and oracle_mod.max_abs_q(q) == qbig
    offs = np.array([0, 3000], np.int64)
    ref, st = oracle_mod.build_hist(bins, 30, sentinel, q, None, offs)
    assert st == oracle_mod.OK and ref[0, :, :, 0].sum(axis=1).max() >= qbig - 3000
    with Session() as s:
        s.upload_bins(bins, 30, sentinel)
        assert g.gbt_begin_tree(s.ctx, gp, 1.0, 1.0e4) == 0
        assert s.sync() == g.GBT_ERR_QUANT_OVERFLOW
        assert s.sync() == 0  # the word was cleared; the context stays usable
        s.begin_tree(np.clip(gp, -1.0, 1.0), 1.0, 1.0e4)
        h = s.build_level(None, offs)
        assert s.sync() == 0
        q2, _ = oracle_mod.quantise(np.clip(gp, -1.0, 1.0), 1.0, 1.0e4)
        ref2, _ = oracle_mod.build_hist(bins, 30, sentinel, q2, None, offs)
        np.testing.assert_array_equal(h.cpu().numpy(), ref2)


def test_determinism_bytes_identical(gb):
    g, Session, s2n = gb
    w = synth.make("level5", n_rows=120_000, n_features=30)
    sg, sh = _scales(w)
    lv = w.levels[5]
    outs = []
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        for _ in range(2):
            hp = s.build_level(w.levels[4].rows, w.levels[4].offsets)
            hs = s.build_level(lv.built_rows, lv.built_offsets)
            large, so, lo = s.subtract_and_find(hp, hs)
            assert s.sync() == 0
            outs.append([x.cpu().numpy().tobytes() for x in (hp, hs, large, so, lo)])
    assert outs[0] == outs[1]


def test_separate_subtract_and_find_match_fused(gb):
    g, Session, s2n = gb
    w = synth.make("level5", n_rows=50_000, n_features=40)
    sg, sh = _scales(w)
    lv = w.levels[5]
    with Session() as s:
        s.upload_bins(w.bins, w.n_bins, w.sentinel).begin_tree(w.gpair, sg, sh)
        hp = s.build_level(w.levels[4].rows, w.levels[4].offsets)
        hs = s.build_level(lv.built_rows, lv.built_offsets)
        large, so, lo = s.subtract_and_find(hp, hs)
        large2 = s.subtract(hp, hs)
        so2 = s.find_splits(hs)
        lo2 = s.find_splits(large2)
        assert s.sync() == 0
        assert torch.equal(large, large2)
        assert torch.equal(so, so2) and torch.equal(lo, lo2)


# --------------------------------------------------------------------------- device error reporting
def test_error_bad_bin_value(gb):
    g, Session, s2n = gb
    bins = np.zeros((2, 100), np.uint8)
    bins[1, 50] = 200  # >= n_bins=10 and not the sentinel
    with Session() as s:
        assert g.gbt_upload_bins(s.ctx, bins, 1, 100, 2, 10, 0xFF) == 0
        assert s.sync() == g.GBT_ERR_BIN_RANGE
        assert s.sync() == 0  # cleared


def test_error_bad_row_and_quant(gb):
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(1, n_rows=100, n_features=2, n_bins=10)
    with Session() as s:
        s.upload_bins(bins, 10, sentinel)
        bad = gp.copy()
        bad[5, 1] = np.inf
        assert g.gbt_begin_tree(s.ctx, bad, 1.0, 1.0) == 0
        assert s.sync() == g.GBT_ERR_QUANT_OVERFLOW
        s.begin_tree(gp, 1.0, 1.0)
        rows = torch.tensor([1, 2, 500], dtype=torch.int32, device="cuda")  # 500 >= n_rows
        offs = torch.tensor([0, 3], dtype=torch.int64, device="cuda")
        h = s.hist_tensor(1)
        assert g.gbt_build_level(s.ctx, rows, offs, 1, h) == 0
        assert s.sync() == g.GBT_ERR_ROW_RANGE
        # host offsets are validated synchronously
        assert g.gbt_build_level(s.ctx, rows, np.array([0, 5, 3], np.int64), 2, s.hist_tensor(2)) == g.GBT_ERR_INVALID_ARG


@pytest.mark.parametrize("width", [1, 2])
@pytest.mark.parametrize("bad_row", [-5, -1, -2 ** 31, 5000])
def test_error_row_outside_range_any_sign(gb, oracle_mod, width, bad_row):
    """A row id outside [0, n_rows), negative ones included, is GBT_ERR_ROW_RANGE at gbt_sync, as the
    oracle reports its row error, through gbt_build_level and gbt_level_step, wherever the id sits in its
    node (first row, last row of a ragged chunk)."""
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(width, n_rows=5000, n_features=70 if width == 1 else 20, n_bins=40, seed=4)
    rng = np.random.default_rng(5)
    rows = rng.permutation(5000)[:3001].astype(np.int32)
    offs = np.array([0, 1200, 3001], np.int64)
    q, _ = oracle_mod.quantise(gp, 1024.0, 1024.0)
    for pos in (0, 1199, 3000):
        bad = rows.copy()
        bad[pos] = bad_row
        _, st = oracle_mod.build_hist(bins, 40, sentinel, q, bad, offs)
        assert st == oracle_mod.ERR_ROW
        with Session() as s:
            s.upload_bins(bins, 40, sentinel).begin_tree(gp, 1024.0, 1024.0)
            hp = s.build_level(None, np.array([0, 2500, 5000], np.int64))
            assert s.sync() == 0
            assert g.gbt_build_level(s.ctx, torch.from_numpy(bad).cuda(), torch.from_numpy(offs).cuda(), 2,
                                     s.hist_tensor(2)) == 0
            assert s.sync() == g.GBT_ERR_ROW_RANGE, (pos, "build")
            hs, large = s.hist_tensor(2), s.hist_tensor(2)
            so = torch.empty((2, g.SPLIT_BYTES), dtype=torch.uint8, device="cuda")
            lo = torch.empty_like(so)
            assert g.gbt_level_step(s.ctx, torch.from_numpy(bad).cuda(), torch.from_numpy(offs).cuda(), 2, hp, None,
                                    hs, large, g.params(1.0, 0.0, 0.0), so, lo) == 0
            assert s.sync() == g.GBT_ERR_ROW_RANGE, (pos, "level step")
            # and the same call on valid rows is clean
            assert g.gbt_build_level(s.ctx, torch.from_numpy(rows).cuda(), torch.from_numpy(offs).cuda(), 2,
                                     s.hist_tensor(2)) == 0
            assert s.sync() == 0


def test_error_inconsistent_subtraction(gb):
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(1, n_rows=100, n_features=2, n_bins=10)
    with Session() as s:
        s.upload_bins(bins, 10, sentinel).begin_tree(gp, 1.0, 100.0)
        hp = s.build_level(None, np.array([0, 50], np.int64))
        hs = s.build_level(None, np.array([0, 100], np.int64))  # "small" larger than parent
        s.subtract(hp, hs)
        assert s.sync() == g.GBT_ERR_INCONSISTENT


def test_error_alloc_fault_injection(gb, monkeypatch):
    """Host-side fault injection: the next allocation fails with GBT_ERR_OOM, the context stays usable."""
    g, Session, s2n = gb
    bins, gp, sentinel = _tiny(1, n_rows=100, n_features=2, n_bins=10)
    big, _, _ = _tiny(1, n_rows=5000, n_features=3, n_bins=10)
    with Session() as s:
        s.upload_bins(bins, 10, sentinel)
        monkeypatch.setenv("GBT_FAULT_ALLOC_AT", "1:first")
        st = g.gbt_upload_bins(s.ctx, big, 1, 5000, 3, 10, 0xFF)  # needs a larger mirror -> allocation 1
        assert st == g.GBT_ERR_OOM, g.gbt_last_error(s.ctx)
        monkeypatch.delenv("GBT_FAULT_ALLOC_AT")
        s.upload_bins(big, 10, 0xFF).begin_tree(np.zeros((5000, 2), np.float32) + 0.5, 2.0, 2.0)
        h = s.build_level(None, np.array([0, 5000], np.int64))
        assert s.sync() == 0
        assert int(h[0, 0, :, 1].sum()) == 5000


# --------------------------------------------------------------------------- split find: golden cases and adversarial ties
def _dummy_session(Session, n_bins, n_features, scale_g=1.0, scale_h=1.0):
    """A context whose dataset shape (features, bins) matches histograms passed in directly."""
    s = Session()
    bins = np.zeros((n_features, 8), np.uint8 if n_bins < 255 else np.uint16)
    s.upload_bins(bins, n_bins, 0xFF if n_bins < 255 else 0xFFFF)
    s.begin_tree(np.zeros((8, 2), np.float32), scale_g, scale_h)
    return s


def test_golden_split_cases_on_gpu(gb):
    """The hand-worked cases of tests/golden/split_cases.json through gbt_find_splits."""
    import json
    import os
    from fractions import Fraction
    g, Session, s2n = gb
    with open(os.path.join(os.path.dirname(__file__), "golden", "split_cases.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        hist = torch.tensor(np.array(case["hist"], np.int64)[None]).cuda()
        s = _dummy_session(Session, case["n_bins"], hist.shape[1])
        try:
            out = s2n(s.find_splits(hist, lam=case["lambda"], gamma=case["gamma"], mcw=case["min_child_weight"]))
            assert s.sync() == 0
        finally:
            s.close()
        e = case["expect"]
        for k in ("feature", "bin", "default_left", "g_left", "h_left", "g_right", "h_right"):
            assert int(out[k][0]) == e[k], (case["name"], k)
        if e["gain"] == "-inf":
            assert out["gain"][0] == -np.inf
        else:
            assert out["gain"][0] == pytest.approx(float(Fraction(e["gain"])), rel=1e-14), case["name"]


@pytest.mark.parametrize("seed,lam,gamma,mcw,sg,sh", [
    (0, 1.0, 0.0, 0.0, 1.0, 1.0),
    (1, 0.0, 0.5, 0.0, 1024.0, 4096.0),
    (2, 3.0, -2.0, 1.5, 2.0 ** 20, 2.0 ** 18),
    (3, 1e-3, 1e3, 0.0, 2.0 ** -20, 2.0 ** -10),   # tiny scales: huge converted values
    (4, 0.0, 0.0, 0.0, 2.0 ** 40, 2.0 ** 40),        # huge scales: tiny converted values (double path)
])
def test_split_find_adversarial_ties_and_ranges(gb, oracle_mod, seed, lam, gamma, mcw, sg, sh):
    """Random histograms with duplicated features (exact ties), magnitudes over many binades, cuts with
    equal gains in both directions; the GPU must match the all-double oracle bit for bit."""
    g, Session, s2n = gb
    rng = np.random.default_rng(900 + seed)
    n_nodes, F, n_bins = 6, 23, 61
    B = n_bins + 1
    hist = np.zeros((n_nodes, F, B, 2), np.int64)
    for n in range(n_nodes):
        for f in range(F):
            scale = 2.0 ** rng.integers(0, 40)
            hist[n, f, :, 0] = (rng.standard_normal(B) * scale).astype(np.int64)
            hist[n, f, :, 1] = (rng.random(B) * scale).astype(np.int64) + 1
            if rng.random() < 0.3:
                hist[n, f, -1] = 0  # no missing mass: both directions tie
        hist[n, 5] = hist[n, 2]        # duplicated features: exact ties across features
        hist[n, 11] = hist[n, 2]
        hist[n, 7, 3:] = 0             # mass concentrated at the start
    out_ref, st = oracle_mod.find_splits(hist, n_bins, lam, gamma, mcw, sg, sh)
    s = _dummy_session(Session, n_bins, F, sg, sh)
    try:
        got = s2n(s.find_splits(torch.from_numpy(hist).cuda(), lam=lam, gamma=gamma, mcw=mcw))
        assert s.sync() == 0
    finally:
        s.close()
    assert_splits_equal(got, out_ref, f"seed {seed}")
