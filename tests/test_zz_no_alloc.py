"""The allocation-free split find, against the oracle and against the context's split find.

Some callers cannot allocate device memory. One example is a host application that hands out all device
memory from its own pool. Another is code that keeps work stream-ordered, where a cudaMalloc would
synchronise the device. gbt_find_splits_noalloc serves them: its scratch is a fixed array inside the
library. This file is collected last, so a failure here cannot hide another GPU test from a run that
stops at the first failure.
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


def _oracle_hists(oracle, w, depths, sg, sh):
    """The oracle's own histograms of the given levels (inputs that never pass through the library)."""
    q, st = oracle.quantise(w.gpair, sg, sh)
    assert st == oracle.OK
    out = []
    for d in depths:
        lv = w.levels[d]
        h, st = oracle.build_hist(w.bins, w.n_bins, w.sentinel, q, lv.rows, lv.offsets)
        assert st == oracle.OK
        out.append(h)
    return out


@pytest.mark.parametrize("name,n_rows,n_features,depths", [
    ("level5", 30_000, 70, (2, 3)),     # u8: 256 slots, strips staged in shared memory
    ("u16miss", 20_000, 11, (3, 2)),    # u16: 4097 slots with 40% missing, strips read from global memory
])
def test_noalloc_matches_oracle_and_context_find_two_calls_in_a_row(oracle_mod, name, n_rows, n_features, depths):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g
    from histogram_construction_gb300.session import Session

    w = synth.make(name, n_rows=n_rows, n_features=n_features, depth=max(depths))
    sg, sh = synth.fixed_point_scales(w.gpair)
    lam, gamma, mcw = 1.0, 0.5, 1e-3
    hists = _oracle_hists(oracle_mod, w, depths, sg, sh)
    refs = [oracle_mod.find_splits(h, w.n_bins, lam, gamma, mcw, sg, sh)[0] for h in hists]
    with Session(0) as sess:
        sess.upload_bins(w.bins, w.n_bins, w.sentinel)
        sess.begin_tree(w.gpair, sg, sh)
        dev = [torch.from_numpy(h).cuda() for h in hists]
        ctx_refs = [_splits(sess.find_splits(h, lam, gamma, mcw)) for h in dev]
        assert sess.sync() == 0
        for r, c in zip(refs, ctx_refs):
            _same(c, r, "context find vs oracle")
        stream = sess.stream.cuda_stream
        prm = g.params(lam, gamma, mcw)
        # two different inputs in a row (the second call runs on whatever the first left in the shared
        # scratch), then the first again
        for call, k in enumerate((0, 1, 0)):
            n = dev[k].shape[0]
            out = torch.zeros((n, g.SPLIT_BYTES), dtype=torch.uint8, device=sess.device)
            st = g.gbt_find_splits_noalloc(dev[k], n, w.n_features, w.n_bins, sg, sh, prm, out, stream)
            assert st == g.GBT_OK, st
            torch.cuda.synchronize()
            _same(_splits(out), refs[k], f"call {call} vs oracle")
            _same(_splits(out), ctx_refs[k], f"call {call} vs context find")


def test_noalloc_allocates_no_device_memory(oracle_mod):
    """After a first call (which may load the library's module on this device), further calls leave the
    device's free memory unchanged."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import histogram_construction_gb300 as g

    w = synth.make("u16miss", n_rows=8_000, n_features=5, depth=2)
    sg, sh = synth.fixed_point_scales(w.gpair)
    (h,) = _oracle_hists(oracle_mod, w, (2,), sg, sh)
    ref, _ = oracle_mod.find_splits(h, w.n_bins, 1.0, 0.0, 0.0, sg, sh)
    hd = torch.from_numpy(h).cuda()
    out = torch.zeros((h.shape[0], g.SPLIT_BYTES), dtype=torch.uint8, device="cuda")
    prm = g.params(1.0, 0.0, 0.0)
    assert g.gbt_find_splits_noalloc(hd, h.shape[0], w.n_features, w.n_bins, sg, sh, prm, out) == g.GBT_OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert g.gbt_find_splits_noalloc(hd, h.shape[0], w.n_features, w.n_bins, sg, sh, prm, out) == g.GBT_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    _same(_splits(out), ref, "after repeated calls")


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
