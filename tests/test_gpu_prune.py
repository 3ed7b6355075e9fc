"""The pruned column blocks of the tensor-core k-NN (pivot bounds, two passes)
change which blocks are evaluated, never the result: on every set below the
tensor-core engine, which prunes once the column set has 16 384 points or
more, returns the same bits as the FP32 engine, which evaluates every block;
sampled rows also agree with the oracle.  The sets cover clustered data with
outliers (the case the bounds are for), data far from the origin (large norms
against small distances), heavy duplication (upper bounds of zero), spread
uniform data, a ragged last block, and queries that differ from the
columns."""

import numpy as np
import pytest

import workloads
from gpu_common import H, dev, np_, oracle_knn_check

pytestmark = pytest.mark.gpu


@pytest.fixture
def h():
    mod = H()
    prev = mod.set_engine("auto")
    yield mod
    mod.set_engine(prev)


def both(h, fn):
    """(FP32 engine result, tensor-core result, tile pairs of the tensor call)."""
    h.set_engine("simt")
    a = fn()
    h.set_engine("tensor")
    b = fn()
    pairs = h.last_knn_tile_pairs()
    h.set_engine("auto")
    return a, b, pairs


def mixture(n, d, seed, clusters=20, outlier_frac=0.05, dup_frac=0.0, mean_sd=4.0):
    return workloads.draw(workloads.Mixture(n=n, d=d, clusters=clusters, mean_sd=mean_sd,
                                            sigma=None, sigma_range=(0.5, 2.0),
                                            outlier_frac=outlier_frac, dup_frac=dup_frac,
                                            seed=seed))


def full_pairs(n, m):
    return ((n + 127) // 128) * ((m + 127) // 128) * 128 * 128


def check_core(h, X, ms, max_frac=None):
    n = X.shape[1]
    a, b, pairs = both(h, lambda: tuple(np_(t) for t in h.core_distances(dev(X), ms)))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
    if max_frac is not None:
        assert pairs <= max_frac * full_pairs(n, n), (pairs, full_pairs(n, n))
    return b


def test_core_pruned_50k_clusters(h):
    """The 50k-clip workload: identical core distances and lists, sampled rows
    against the oracle, and most blocks pruned."""
    X, task = workloads.workload("hdbscan_50k_d61")
    ms = task["min_samples"]
    core, idx, dist = check_core(h, X, ms, max_frac=0.6)
    rows = np.random.default_rng(0).choice(X.shape[1], 300, replace=False)
    oracle_knn_check(X, X, ms + 1, idx, dist, rows=rows, where="pruned core 50k")


def test_core_pruned_far_from_origin(h):
    """Norms ~1e4 times the neighbour distances: the ranking proof and the
    pruning bounds both work near their rounding limits."""
    X = mixture(20000, 32, seed=11) + np.float32(300.0)
    check_core(h, np.ascontiguousarray(X, dtype=np.float32), 7)


def test_core_pruned_heavy_duplicates(h):
    """Every point has many exact copies: k-th distances (and upper bounds) of 0."""
    rng = np.random.default_rng(4)
    base = mixture(400, 24, seed=5, outlier_frac=0.0)
    X = np.ascontiguousarray(base[:, rng.integers(0, 400, size=24000)])
    check_core(h, X, 10)


def test_core_pruned_uniform_low_dim(h):
    """Uniform points in a 6-dimensional cube: no clusters."""
    X = np.random.default_rng(6).uniform(-1, 1, size=(6, 30000)).astype(np.float32)
    check_core(h, X, 5)


def test_core_pruned_ragged_tail(h):
    """One column past a whole number of blocks (the last block holds one point)."""
    X = mixture(16385, 61, seed=9)
    check_core(h, X, 10)


@pytest.mark.parametrize("n,m,d,k", [(30000, 20000, 40, 10), (5000, 17000, 64, 16),
                                     (20001, 16384, 17, 32)])
def test_knn_pruned_queries_differ(h, n, m, d, k):
    """Queries that are not the columns (the home blocks come from the bins'
    matching positions): identical to the FP32 engine, sampled rows against
    the oracle."""
    X = mixture(n, d, seed=n + d)
    Y = mixture(m, d, seed=m + 7 * d)
    (ai, ad), (bi, bd), pairs = both(h, lambda: tuple(np_(t) for t in h.knn(dev(X), dev(Y), k)))
    assert np.array_equal(ai, bi) and np.array_equal(ad, bd)
    assert pairs <= full_pairs(n, m)
    rows = np.random.default_rng(1).choice(n, 200, replace=False)
    oracle_knn_check(X, Y, k, bi, bd, rows=rows, where=f"pruned knn n={n} m={m} d={d}")
