"""Mutual-reachability MST on the GPU against the float64 oracle (Prim)."""

import numpy as np
import pytest

import goldens
import oracle
import oracle_pins
import parity
import workloads
from gpu_common import H, dev, golden_outputs, golden_total, np_

pytestmark = pytest.mark.gpu


def gpu_tree(h, X, ms, shortcuts=True):
    Xd = dev(X)
    core, idx, dist = h.core_distances(Xd, ms)
    if shortcuts:
        edges, w = h.mr_mst(Xd, core, idx, dist)
    else:
        edges, w = h.mr_mst(Xd, core)
    e = np_(edges)
    return np_(core), e[:, 0].astype(np.int64), e[:, 1].astype(np.int64), np_(w)


def full_check(h, X, ms, where, shortcuts=True):
    core, lo, hi, w = gpu_tree(h, X, ms, shortcuts)
    oc = oracle.core_distances(X, ms)
    parity.check_core(core, oc, where=where)
    olo, ohi, ow = oracle.prim_mst(X, oc)
    floor = 1e-5 * float(np.median(oc))
    return parity.check_mst(X.shape[1], lo, hi, w, olo, ohi, ow,
                            lambda a, b: oracle.mr_weights(X, oc, a, b), floor, where=where)


@pytest.mark.parametrize("shortcuts", [True, False])
@pytest.mark.parametrize("g", goldens.all_fixtures(), ids=lambda g: g["name"])
def test_mst_golden(g, shortcuts):
    """Hand-worked trees, exact ties included: the edges must be exactly those."""
    h = H()
    core, lo, hi, w = gpu_tree(h, g["X"], g["min_samples"], shortcuts)
    assert [(int(a), int(b)) for a, b in zip(lo, hi)] == [(a, b) for a, b, _ in g["edges"]]
    assert np.allclose(w, [c for _, _, c in g["edges"]], rtol=1e-6, atol=0)


@pytest.mark.parametrize("shortcuts", [True, False])
@pytest.mark.parametrize("n,d,ms", [(2, 1, 1), (3, 2, 2), (5, 61, 2), (127, 61, 10), (129, 3, 5),
                                    (300, 64, 1), (1001, 65, 7), (1500, 102, 10)])
def test_mst_ragged(n, d, ms, shortcuts):
    h = H()
    X = workloads.small(n, d, seed=n * 3 + d, dup_frac=0.05, outlier_frac=0.05)
    full_check(h, X, ms, f"n={n} d={d} ms={ms} shortcuts={shortcuts}", shortcuts)


@pytest.mark.parametrize("seed,n,d,ms", [(1, 200, 2, 3), (2, 500, 3, 5), (3, 1000, 4, 10),
                                         (4, 130, 1, 2), (5, 700, 6, 1)])
def test_mst_integer_points_exact(seed, n, d, ms):
    """Integer coordinates: weights are exact on both sides, so the tree (ties
    included) must be the oracle's tree edge for edge."""
    h = H()
    rng = np.random.default_rng(seed)
    X = oracle_pins.int_points(rng, n, d, span=3, dup_frac=0.2)
    for shortcuts in (True, False):
        core, lo, hi, w = gpu_tree(h, X, ms, shortcuts)
        oc = oracle.core_distances(X, ms)
        olo, ohi, ow = oracle.prim_mst(X, oc)
        assert np.array_equal(lo, olo) and np.array_equal(hi, ohi), (shortcuts,)
        assert np.array_equal(w.astype(np.float64), ow.astype(np.float32).astype(np.float64))


@pytest.mark.parametrize("name", ["hdbscan_2k_d61"])
def test_mst_2k_d61(name):
    h = H()
    X, task = workloads.workload(name)
    full_check(h, X, task["min_samples"], name)
    g = golden_total(name, X)
    _, _, _, w = gpu_tree(h, X, task["min_samples"])
    assert abs(w.astype(np.float64).sum() - g["mst_total"]) <= 1e-5 * g["mst_total"]


def test_mst_50k_d61():
    h = H()
    X, task = workloads.workload("hdbscan_50k_d61")
    full_check(h, X, task["min_samples"], "50k")


def test_pruning_is_exact():
    """The shortcuts change no bit of the tree (page "HDBSCAN", "Exact shortcuts":
    the tree built both ways on clip-like data with duplicates is identical)."""
    h = H()
    sets = [workloads.workload("hdbscan_2k_d61")[0],
            workloads.small(3000, 61, seed=17, dup_frac=0.05, outlier_frac=0.1),
            np.ascontiguousarray(np.repeat(workloads.small(100, 8, seed=3), 7, axis=1))]
    for X in sets:
        for ms in (2, 5, 10):
            a = gpu_tree(h, X, ms, True)
            b = gpu_tree(h, X, ms, False)
            for u, v in zip(a, b):
                assert np.array_equal(u, v)


def test_mst_all_points_identical():
    """Every weight is 0: the (w, lo, hi) order makes the tree the star at point 0."""
    h = H()
    X = np.ones((5, 257), dtype=np.float32)
    core, lo, hi, w = gpu_tree(h, X, 3)
    assert (lo == 0).all() and np.array_equal(hi, np.arange(1, 257)) and (w == 0).all()


def test_mst_single_point():
    h = H()
    X = np.zeros((4, 1), dtype=np.float32)
    core, lo, hi, w = gpu_tree(h, X, 1)
    assert lo.shape == (0,) and w.shape == (0,)


def test_mst_bad_core_rejected():
    h = H()
    X = workloads.small(100, 8, seed=2)
    core = np.ones(100, dtype=np.float32)
    core[5] = np.inf
    with pytest.raises(h.HdbmstError) as e:
        h.mr_mst(dev(X), dev(core))
    assert e.value.status == 4


def test_mst_200k_d61_bench_config():
    """The benchmark's workload at full size, in its launch configuration,
    against the oracle's whole output (stored by make_oracle_totals.py from
    the oracle alone): every core distance, and the whole tree by the parity
    rules (structure, per-edge weights, total, and every edge on one side only
    a near-tie exchange in both directions: page "HDBSCAN", "A lesson about
    tests: ties")."""
    h = H()
    X, task = workloads.workload("hdbscan_200k_d61")
    ms = task["min_samples"]
    n = X.shape[1]
    g = golden_outputs("hdbscan_200k_d61", X)
    assert int(g["min_samples"]) == ms
    core, lo, hi, w = gpu_tree(h, X, ms)
    oc = g["core"]
    parity.check_core(core, oc, where="200k x 61 cores")
    floor = 1e-5 * float(np.median(oc))
    olo, ohi = g["lo"].astype(np.int64), g["hi"].astype(np.int64)
    ow = oracle.mr_weights(X, oc, olo, ohi)
    exchanged = parity.check_mst(n, lo, hi, w, olo, ohi, ow,
                                 lambda a, b: oracle.mr_weights(X, oc, a, b), floor,
                                 where="200k x 61 tree")
    tot = golden_total("hdbscan_200k_d61", X)["mst_total"]
    assert np.sum(ow) == tot
    print(f"200k x 61: {exchanged} near-tie exchanges against the oracle tree")
