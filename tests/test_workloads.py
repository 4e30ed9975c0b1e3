"""The seeded workload generators draw what their docstring promises (host only)."""
import os

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


def _page_shapes():
    """Geometries and token counts from ``tests/golden/page_workload_shapes.txt``."""
    geometry, tokens = {}, {}
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "page_workload_shapes.txt")
    with open(path) as f:
        for line in f:
            fields = line.split("#", 1)[0].split()
            if not fields:
                continue
            if fields[0] == "geometry":
                geometry[fields[1]] = tuple(int(v) for v in fields[2:6])
            elif fields[0] == "tokens":
                tokens[fields[1]] = {int(v) for v in fields[2:]}
    return geometry, tokens


def test_shapes_follow_the_pages():
    """The decode, prefill and Zipf small-batch workloads use the expert
    geometries the DeepGEMM and FlashInfer pages benchmark, at token counts
    the DeepGEMM page times. (tiny is a small parity case; large is a
    hot-expert case at its own geometry: 128 experts, top-8, 4096 / 1536.)"""
    geometry, tokens = _page_shapes()
    shape = {name: (wl.E, wl.k, wl.H, wl.I) for name, wl in wlm.WORKLOADS.items()}
    for name in ("decode1", "decode8", "prefill"):
        assert shape[name] == geometry["deepgemm"], name
    assert shape["small"] == geometry["flashinfer"]
    for name in ("decode1", "decode8", "small", "prefill", "large"):
        assert wlm.WORKLOADS[name].T in tokens["deepgemm"], name
