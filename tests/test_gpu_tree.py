"""A whole depth-wise tree on the device, level by level, against the oracle's own tree.

Every level after the root runs two calls: gbt_partition_level_pairs routes the rows by the previous
level's splits and lists each pair's smaller child, and gbt_advance_level builds those, derives their
siblings and finds every node's split, in node order (bonsai '10: CUDA histogram backend', 'The device
context lifecycle': partition_level, advance_level). The oracle grows the same tree from its own
histograms and splits with its serial partition; rows, offsets, smaller-child lists, histograms and
splits are compared bit for bit at every level.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _oracle_levels(oracle, w, sg, sh, depth, lam, gamma, mcw):
    """Yields, per level, the oracle's (rows, offsets, small_side, small_offsets, small_rows, hist, splits)."""
    q, st = oracle.quantise(w.gpair, sg, sh)
    assert st == oracle.OK
    N = w.n_rows
    offs = np.array([0, N], np.int64)
    h, st = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, None, offs)
    assert st == oracle.OK
    sp, _ = oracle.find_splits(h, w.n_bins, lam, gamma, mcw, sg, sh)
    rows = None
    yield None, offs, None, None, None, h, sp
    for _ in range(depth):
        rows, offs, st = oracle.partition(w.bins, w.n_bins, w.sentinel, rows, offs, sp)
        assert st == oracle.OK
        sizes = np.diff(offs)
        n = sizes.shape[0]
        side = (sizes[1::2] < sizes[0::2]).astype(np.uint8)  # the smaller child; ties go left
        small = np.arange(0, n, 2) + side
        b_rows = np.concatenate([rows[offs[i]:offs[i + 1]] for i in small]).astype(np.int32)
        b_offs = np.concatenate([[0], np.cumsum(sizes[small])]).astype(np.int64)
        hs, st = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, b_rows, b_offs)
        assert st == oracle.OK
        hl, st = oracle.subtract(h, None, hs)
        assert st == oracle.OK
        h = np.empty((n,) + hs.shape[1:], np.int64)
        h[small] = hs
        h[small ^ 1] = hl
        del hs, hl
        sp, _ = oracle.find_splits(h, w.n_bins, lam, gamma, mcw, sg, sh)
        yield rows, offs, side, b_offs, b_rows, h, sp


def _same_splits(got, ref, where):
    for k in ("feature", "bin", "default_left", "g_left", "h_left", "g_right", "h_right"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=f"{where} field {k}")
    np.testing.assert_array_equal(got["gain"].view(np.int64), ref["gain"].view(np.int64), err_msg=f"{where} gain")


def _grow_and_compare(oracle, w, depth, lam=1.0, gamma=0.0, mcw=0.0):
    from histogram_construction_gb300.session import Session, splits_to_numpy
    sg, sh = synth.fixed_point_scales(w.gpair)
    N = w.n_rows
    ref = _oracle_levels(oracle, w, sg, sh, depth, lam, gamma, mcw)
    with Session() as s:
        s.upload_bins(torch.from_numpy(w.bins).cuda(), w.n_bins, w.sentinel)
        s.begin_tree(torch.from_numpy(w.gpair).cuda(), sg, sh)
        offs_d = torch.tensor([0, N], dtype=torch.int64, device="cuda")
        h_d = s.build_level(None, offs_d)
        sp_d = s.find_splits(h_d, lam, gamma, mcw)
        _, _, _, _, _, h_ref, sp_ref = next(ref)
        assert s.sync() == 0
        np.testing.assert_array_equal(h_d.cpu().numpy(), h_ref, err_msg="root hist")
        _same_splits(splits_to_numpy(sp_d), sp_ref, "root")
        rows_d = None
        for d in range(1, depth + 1):
            rows_d, offs_d, srows_d, soffs_d, sside_d = s.partition_pairs(rows_d, offs_d, sp_d, n_rows_level=N)
            h_d, sp_d = s.advance_level(srows_d, soffs_d, sside_d, h_d, lam=lam, gamma=gamma, mcw=mcw)
            assert s.sync() == 0, f"level {d}"
            rows, offs, side, b_offs, b_rows, h_ref, sp_ref = next(ref)
            np.testing.assert_array_equal(offs_d.cpu().numpy(), offs, err_msg=f"offsets level {d}")
            np.testing.assert_array_equal(rows_d.cpu().numpy(), rows, err_msg=f"rows level {d}")
            np.testing.assert_array_equal(sside_d.cpu().numpy(), side, err_msg=f"small side level {d}")
            np.testing.assert_array_equal(soffs_d.cpu().numpy(), b_offs, err_msg=f"small offsets level {d}")
            np.testing.assert_array_equal(srows_d[:b_rows.shape[0]].cpu().numpy(), b_rows,
                                          err_msg=f"small rows level {d}")
            np.testing.assert_array_equal(h_d.cpu().numpy(), h_ref, err_msg=f"hist level {d}")
            _same_splits(splits_to_numpy(sp_d), sp_ref, f"splits level {d}")


def test_tree_dense_reduced_all_levels(oracle_mod):
    """The dense workload's shape at 150,000 x 130 (a ragged second feature tile), constant h, levels 0..7."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synth.make("dense", n_rows=150_000, n_features=130, depth=0)
    _grow_and_compare(oracle_mod, w, 7, lam=1.0, mcw=0.5)


def test_tree_u16_missing_reduced(oracle_mod):
    """u16 bins with 40% missing (the missing direction decides routing), levels 0..6."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synth.make("u16miss", n_rows=80_000, n_features=21, depth=0)
    _grow_and_compare(oracle_mod, w, 6, lam=0.5, gamma=0.1)


def test_tree_dense_full_size_all_levels(oracle_mod):
    """10,000,000 x 500 u8, h = 0.25: the depth-8 tree (levels 0..7) of the benchmark, compared in full."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = synth.make("dense", depth=0)
    _grow_and_compare(oracle_mod, w, 7)
