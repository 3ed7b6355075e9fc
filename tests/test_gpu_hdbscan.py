"""The whole method on the GPU plus the host back half: labels against the
oracle's back half (oracle/hierarchy.py).

On the spanning tree the GPU produced, the library's labels must equal the
oracle's bit for bit (same tree, same definitions).  Against the oracle's own
float64 Prim tree the labels may differ only where the trees differ at tied
weights (page "HDBSCAN", "A lesson about tests: ties"); min_cluster_size = 20
as in the page's "Results"."""

import numpy as np
import pytest

import goldens
import oracle
from oracle import hierarchy
import oracle_pins
import workloads
from gpu_common import H, dev

pytestmark = pytest.mark.gpu

MCS = 20


def _gpu(X, ms, mcs):
    h = H()
    labels, core, edges, w = h.hdbscan(dev(X), ms, mcs)
    return labels, core, edges, w


def test_golden_labels_gpu():
    for g in goldens.all_fixtures():
        if "labels" not in g:
            continue
        labels, _, _, _ = _gpu(g["X"], g["min_samples"], g["min_cluster_size"])
        assert np.array_equal(labels, g["labels"]), g["name"]


@pytest.mark.parametrize("name", ["hdbscan_2k_d61", "hdbscan_50k_d61", "hdbscan_200k_d61"])
def test_labels_equal_oracle_back_half_on_gpu_tree(name):
    X, task = workloads.workload(name)
    labels, core, edges, w = _gpu(X, task["min_samples"], MCS)
    n = X.shape[1]
    want = hierarchy.hdbscan_labels(n, edges[:, 0], edges[:, 1], w, MCS)
    assert np.array_equal(labels, want)
    assert len(set(labels.tolist()) - {-1}) >= 2, "the mixture yields several clusters"


def test_labels_against_oracle_prim_2k():
    """Oracle core distances and float64 Prim tree, oracle back half: the same
    clusters, except at most 1% of points (ties)."""
    X, task = workloads.workload("hdbscan_2k_d61")
    ms = task["min_samples"]
    labels, _, _, _ = _gpu(X, ms, MCS)
    o = oracle.default()
    lo, hi, w = o.prim_mst(X, o.core_distances(X, ms))
    want = hierarchy.hdbscan_labels(X.shape[1], lo, hi, w, MCS)
    assert len(set(labels.tolist())) == len(set(want.tolist()))
    mapped = np.full(labels.shape, -1)
    for c in set(labels.tolist()) - {-1}:
        vals, cnt = np.unique(want[labels == c], return_counts=True)
        mapped[labels == c] = vals[np.argmax(cnt)]
    assert np.mean(mapped != want) <= 0.01


def test_labels_integer_points_exact():
    """Integer coordinates: every weight is exact, the trees are identical,
    so are the labels."""
    rng = np.random.default_rng(41)
    X = oracle_pins.int_points(rng, 600, 3, span=12, dup_frac=0.05)
    labels, _, _, _ = _gpu(X, 4, 10)
    o = oracle.default()
    lo, hi, w = o.prim_mst(X, o.core_distances(X, 4))
    want = hierarchy.hdbscan_labels(600, lo, hi, w, 10)
    assert np.array_equal(labels, want)
