"""The synthetic input recipe: seeded determinism, and the structure each
workload description asks for (radius graphs: mean in-degree about 32,
symmetric edges without self-loops, edge vectors shorter than the radius,
cell-ordered node labels so neighbours have nearby indices; the Poisson graph:
in-degree mean 32 and uniform sources; weight scales N(0,1)/sqrt(P) or N(0,1))."""
import math

import numpy as np
import pytest

from oracle import tp
from workloads import WORKLOADS, make_features, make_graph


def test_seeded_and_reproducible():
    wl = WORKLOADS["medium"]
    a = make_graph(wl, 0)
    b = make_graph(wl, 0)
    c = make_graph(wl, 1)
    for u, v in zip(a[1:4], b[1:4]):
        np.testing.assert_array_equal(u, v)
    assert len(a[1]) != len(c[1]) or not np.array_equal(a[1], c[1])


@pytest.mark.parametrize("name", ["medium", "xlarge"])
def test_radius_graphs(name):
    wl = WORKLOADS[name]
    _, src, dst, vec, n = make_graph(wl, 0)
    E = len(src)
    assert n == wl.n_nodes
    assert 30.0 < E / n < 34.0                       # mean degree ~32
    assert np.all(src != dst) and np.all(np.diff(dst) >= 0)
    r = np.linalg.norm(vec, axis=1)
    assert np.all(r > 0) and np.all(r < wl.radius)
    # symmetric: j -> i exists exactly when i -> j does
    fwd = np.sort(src.astype(np.int64) * n + dst)
    bwd = np.sort(dst.astype(np.int64) * n + src)
    np.testing.assert_array_equal(fwd, bwd)
    # the reverse edge's vector is the negated one (minimum image)
    key = src.astype(np.int64) * n + dst
    order = np.argsort(key)
    rev = order[np.searchsorted(key[order], dst.astype(np.int64) * n + src)]
    np.testing.assert_allclose(vec[rev], -vec, atol=1e-9)
    # cell-ordered labels: neighbours sit close in index compared with n
    assert np.median(np.abs(src.astype(np.int64) - dst)) < n / 8


def test_poisson_graph():
    wl = WORKLOADS["large"]
    _, src, dst, vec, n = make_graph(wl, 0)
    deg = np.bincount(dst, minlength=n)
    assert abs(deg.mean() - 32.0) < 0.2 and abs(deg.var() - 32.0) < 1.5   # Poisson(32)
    assert src.min() >= 0 and src.max() < n and np.all(np.diff(dst) >= 0)
    assert abs(src.mean() / n - 0.5) < 0.01                                  # uniform sources
    np.testing.assert_allclose(np.linalg.norm(vec, axis=1), 1.0, rtol=1e-12)


@pytest.mark.parametrize("name,scaled", [("medium", True), ("large", True), ("xlarge", False)])
def test_feature_scales(name, scaled):
    wl = WORKLOADS[name]
    pl = tp.Plan(wl.irreps_in, wl.irreps_sh, wl.irreps_out)
    rng = np.random.default_rng(3)
    x, w, _ = make_features(rng, wl, 256, 512, pl.dim_in, pl.weight_numel, pl.n_paths, pl.dim_out)
    assert abs(x.std() - 1.0) < 0.02
    want = 1.0 / math.sqrt(pl.n_paths) if scaled else 1.0
    assert abs(w.std() / want - 1.0) < 0.03
