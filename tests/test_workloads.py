"""The seeded workload generators draw what their docstring promises (host only)."""
import numpy as np
import pytest

import workloads as wlm


@pytest.mark.parametrize("name", list(wlm.WORKLOADS))
def test_routing_shape_and_distinct(name):
    wl = wlm.WORKLOADS[name]
    ids, w = wlm.make_routing(wl)
    assert ids.shape == (wl.T, wl.k) and ids.dtype == np.int32
    assert w.shape == (wl.T, wl.k) and w.dtype == np.float32
    assert ids.min() >= 0 and ids.max() < wl.E
    for row in ids:
        assert len(set(row.tolist())) == wl.k
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-5)
    assert np.all(w > 0)
    ids2, w2 = wlm.make_routing(wl)
    assert np.array_equal(ids, ids2) and np.array_equal(w, w2)


def test_zipf_skew_leaves_empty_experts():
    wl = wlm.WORKLOADS["small"]
    ids, _ = wlm.make_routing(wl)
    counts = np.bincount(ids.reshape(-1), minlength=wl.E)
    assert (counts == 0).sum() >= 40          # several experts get no rows
    assert counts.max() >= 60                 # a few get many
    assert counts[0] == counts.max()          # popularity falls with the expert id


def test_hot_expert_share():
    wl = wlm.WORKLOADS["large"]
    ids, _ = wlm.make_routing(wl)
    hot = ids[:, 0] == 0
    assert hot.sum() >= wl.T // 4
    counts = np.bincount(ids.reshape(-1), minlength=wl.E)
    mean_other = counts[1:].mean()
    assert counts[0] > 4 * mean_other


def test_token_subset():
    wl = wlm.WORKLOADS["prefill"]
    a = wlm.token_subset(wl)
    b = wlm.token_subset(wl)
    assert a.size == 256 and np.array_equal(a, b) and len(set(a.tolist())) == 256
    assert wlm.token_subset(wlm.WORKLOADS["tiny"]).size == wlm.WORKLOADS["tiny"].T


def test_weights_small_shape():
    wl = wlm.custom("t", 4, 3, 2, 64, 32)
    W13, W2 = wlm.make_weights(wl)
    assert W13.shape == (3, 64, 64) and W2.shape == (3, 64, 32)
    assert 0.015 < float(W13.float().std()) < 0.025
    x = wlm.make_x(wl)
    assert x.shape == (4, 64)
