"""The library's HDBSCAN back half (hdbmst_hdbscan_labels, host code) against
the oracle's (oracle/hierarchy.py).  No GPU: the function runs on the host,
so these tests give it spanning trees made by the oracle or drawn at random
and require identical labels."""

import numpy as np
import pytest

import goldens
import oracle
from oracle import hierarchy
import hdbscan_mst_gb300 as H


def _lib_labels(lo, hi, w, mcs):
    E = np.stack([np.asarray(lo), np.asarray(hi)], 1).astype(np.int32)
    return H.hdbscan_labels(E, np.asarray(w, dtype=np.float32), mcs)


def _random_tree(rng, n, ties=False):
    """A random spanning tree with weights, edges in (w, lo, hi) order."""
    a = np.arange(1, n)
    b = np.array([rng.integers(0, i) for i in range(1, n)])
    lo, hi = np.minimum(a, b), np.maximum(a, b)
    w = rng.integers(1, 8, size=n - 1) if ties else rng.random(n - 1) * 10
    w = np.asarray(w, dtype=np.float32)
    order = np.lexsort((hi, lo, w))
    return lo[order], hi[order], w[order]


def test_golden_labels():
    o = oracle.default()
    for g in goldens.all_fixtures():
        if "labels" not in g:
            continue
        core = o.core_distances(g["X"], g["min_samples"])
        lo, hi, w = o.prim_mst(g["X"], core)
        assert np.array_equal(_lib_labels(lo, hi, w, g["min_cluster_size"]), g["labels"]), g["name"]


@pytest.mark.parametrize("n,d,ms,mcs", [(400, 2, 5, 10), (2000, 8, 5, 15), (1500, 61, 3, 10),
                                        (900, 3, 1, 5), (700, 4, 10, 50)])
def test_oracle_trees(n, d, ms, mcs):
    """Spanning trees of clustered points (oracle core distances and Prim)."""
    rng = np.random.default_rng(n + d)
    P = rng.normal(size=(n, d)) + rng.integers(0, 6, size=(n, 1)) * 4.0
    P[: n // 25] = rng.uniform(P.min(0), P.max(0), size=(n // 25, d))
    X = np.ascontiguousarray(P.astype(np.float32).T)
    o = oracle.default()
    lo, hi, w = o.prim_mst(X, o.core_distances(X, ms))
    w32 = w.astype(np.float32)
    want = hierarchy.hdbscan_labels(n, lo, hi, w32, mcs)
    assert np.array_equal(_lib_labels(lo, hi, w32, mcs), want)


@pytest.mark.parametrize("n,ties,mcs", [(2, False, 2), (3, True, 2), (50, True, 3),
                                        (5000, False, 20), (5000, True, 7), (100000, False, 30)])
def test_random_trees(n, ties, mcs):
    """Arbitrary spanning trees, with and without equal weights."""
    rng = np.random.default_rng(n * 7 + ties)
    lo, hi, w = _random_tree(rng, n, ties)
    want = hierarchy.hdbscan_labels(n, lo, hi, w, mcs)
    assert np.array_equal(_lib_labels(lo, hi, w, mcs), want)


def test_zero_weights_give_infinite_lambda():
    """Exact duplicates at min_samples = 1 merge at weight 0 (lambda infinite)."""
    lo = np.array([0, 1, 2, 4, 5, 3], dtype=np.int64)
    hi = np.array([1, 2, 3, 5, 6, 4], dtype=np.int64)
    w = np.array([0, 0, 0, 0, 0, 7], dtype=np.float32)
    want = hierarchy.hdbscan_labels(7, lo, hi, w, 3)
    assert np.array_equal(_lib_labels(lo, hi, w, 3), want)


def test_small_and_invalid_inputs():
    L = H.lib()
    assert H.hdbscan_labels(np.zeros((0, 2), np.int32), np.zeros(0, np.float32), 2).tolist() == [-1]
    lab = np.empty(3, dtype=np.int32)
    # a cycle: (0,1) twice
    E = np.array([[0, 1], [0, 1]], dtype=np.int32)
    W = np.array([1, 2], dtype=np.float32)
    assert L.hdbmst_hdbscan_labels(E.ctypes.data, W.ctypes.data, 3, 2, lab.ctypes.data) == 1
    # an index out of range
    E = np.array([[0, 1], [1, 3]], dtype=np.int32)
    assert L.hdbmst_hdbscan_labels(E.ctypes.data, W.ctypes.data, 3, 2, lab.ctypes.data) == 1
    # a NaN and a negative weight
    E = np.array([[0, 1], [1, 2]], dtype=np.int32)
    for bad in (np.nan, -1.0, np.inf):
        W = np.array([1, bad], dtype=np.float32)
        assert L.hdbmst_hdbscan_labels(E.ctypes.data, W.ctypes.data, 3, 2, lab.ctypes.data) == 4
    # min_cluster_size below 2
    W = np.array([1, 2], dtype=np.float32)
    assert L.hdbmst_hdbscan_labels(E.ctypes.data, W.ctypes.data, 3, 1, lab.ctypes.data) == 1
