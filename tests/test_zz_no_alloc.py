"""The allocation-free split find against the context's split find.

Some callers cannot allocate device memory. One example is a host application
that hands out all device memory from its own pool. Another is code that keeps
work stream-ordered, where a cudaMalloc would synchronise the device.
gbt_find_splits_noalloc serves them: its scratch is a fixed array inside the
library. This file is collected last, so a failure here cannot hide another
GPU test from a run that stops at the first failure.
"""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _splits(t):
    from histogram_construction_gb300.session import splits_to_numpy
    return splits_to_numpy(t)


def _same(a, b, where):
    for k in ("feature", "bin", "default_left", "g_left", "h_left", "g_right", "h_right"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=f"{where} field {k}")
    np.testing.assert_array_equal(a["gain"].view(np.int64), b["gain"].view(np.int64), err_msg=f"{where} gain")


def test_noalloc_matches_context_find_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g
    from histogram_construction_gb300.session import Session

    w = synth.make("level5", n_rows=30_000, n_features=70, depth=3)
    mg = float(np.abs(w.gpair[:, 0]).max())
    mh = float(np.abs(w.gpair[:, 1]).max())
    s, sg, sh = g.gbt_suggest_scales(0, mg, mh)
    assert s == 0
    lam, gamma, mcw = 1.0, 0.5, 1e-3
    with Session(0) as sess:
        sess.upload_bins(w.bins, w.n_bins, w.sentinel)
        sess.begin_tree(w.gpair, sg, sh)
        # two different inputs: 4 nodes, then 8 nodes (the second call runs on
        # whatever the first left in the shared scratch)
        hists = []
        for depth in (2, 3):
            lv = w.levels[depth]
            hists.append(sess.build_level(lv.rows, torch.from_numpy(lv.offsets).cuda()))
        refs = [_splits(sess.find_splits(h, lam, gamma, mcw)) for h in hists]
        assert sess.sync() == 0
        stream = sess.stream.cuda_stream
        prm = g.params(lam, gamma, mcw)
        for call, h in enumerate(hists):
            n = h.shape[0]
            out = torch.zeros((n, g.SPLIT_BYTES), dtype=torch.uint8, device=sess.device)
            st = g.gbt_find_splits_noalloc(h, n, w.n_features, w.n_bins, sg, sh, prm, out, stream)
            assert st == g.GBT_OK, st
            torch.cuda.synchronize()
            _same(_splits(out), refs[call], f"call {call}")
        # the same input again after a larger call: the counters were cleared
        out = torch.zeros((hists[0].shape[0], g.SPLIT_BYTES), dtype=torch.uint8, device=sess.device)
        assert g.gbt_find_splits_noalloc(hists[0], hists[0].shape[0], w.n_features, w.n_bins, sg, sh, prm, out,
                                         stream) == g.GBT_OK
        torch.cuda.synchronize()
        _same(_splits(out), refs[0], "repeat")


def test_noalloc_rejects_sizes_beyond_its_scratch_and_host_outputs():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g

    prm = g.params(1.0, 0.0, 0.0)
    hist = torch.zeros((1, 16, 256, 2), dtype=torch.int64, device="cuda")
    out = torch.zeros((4097, g.SPLIT_BYTES), dtype=torch.uint8, device="cuda")
    # more nodes than the scratch holds counters for
    assert g.gbt_find_splits_noalloc(hist, 4097, 16, 255, 1.0, 1.0, prm, out) == g.GBT_ERR_UNSUPPORTED
    # more candidates than the scratch holds: 1024 nodes x ceil(300 / 8) = 38,912 > 32,768
    assert g.gbt_find_splits_noalloc(hist, 1024, 300, 255, 1.0, 1.0, prm, out) == g.GBT_ERR_UNSUPPORTED
    # host output would need a staging allocation
    host_out = np.zeros((1, g.SPLIT_BYTES), dtype=np.uint8)
    assert g.gbt_find_splits_noalloc(hist, 1, 16, 255, 1.0, 1.0, prm, host_out) == g.GBT_ERR_INVALID_ARG
    assert g.gbt_find_splits_noalloc(hist, 1, 16, 255, 0.0, 1.0, prm, out) == g.GBT_ERR_INVALID_ARG
