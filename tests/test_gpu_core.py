"""Core distances on the GPU against the float64 oracle."""

import numpy as np
import pytest

import goldens
import oracle
import parity
import workloads
from gpu_common import H, dev, golden_outputs, np_

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("g", goldens.all_fixtures(), ids=lambda g: g["name"])
def test_core_golden(g):
    h = H()
    core, idx, dist = h.core_distances(dev(g["X"]), g["min_samples"])
    assert np.allclose(np_(core), g["core"], rtol=1e-6, atol=0)


@pytest.mark.parametrize("n,d,ms", [(1, 3, 1), (2, 1, 2), (3, 5, 2), (5, 61, 5), (127, 61, 10),
                                    (129, 64, 10), (1001, 65, 7), (2000, 192, 31), (700, 3, 10)])
def test_core_ragged(n, d, ms):
    h = H()
    X = workloads.small(n, d, seed=n + d, dup_frac=0.05)
    core, idx, dist = h.core_distances(dev(X), ms)
    parity.check_core(np_(core), oracle.core_distances(X, ms), where=f"n={n} d={d} ms={ms}")
    L = min(ms + 1, n)
    assert idx.shape == (n, L)
    # the lists are the k-NN of X against itself, bit for bit
    ki, kd = h.knn(dev(X), dev(X), L)
    assert np.array_equal(np_(ki), np_(idx)) and np.array_equal(np_(kd), np_(dist))
    assert np.array_equal(np_(dist)[:, ms - 1], np_(core))


def test_core_min_samples_one_is_zero():
    h = H()
    X = workloads.small(300, 10, seed=1)
    core = h.core_distances(dev(X), 1, lists=False)
    assert (np_(core) == 0).all()


def test_core_min_samples_n_is_farthest():
    h = H()
    X = workloads.small(31, 7, seed=2)
    core = h.core_distances(dev(X), 31, lists=False)
    parity.check_core(np_(core), oracle.core_distances(X, 31))


def test_core_min_samples_beyond_limit():
    h = H()
    X = workloads.small(60, 7, seed=2)
    with pytest.raises(h.HdbmstError) as e:
        h.core_distances(dev(X), 40, lists=False)
    assert e.value.status == 2


def test_core_2k_d61():
    h = H()
    X, task = workloads.workload("hdbscan_2k_d61")
    core = h.core_distances(dev(X), task["min_samples"], lists=False)
    parity.check_core(np_(core), oracle.core_distances(X, task["min_samples"]), where="2k")


def test_core_200k_d61():
    """Every core distance of the 200 000-clip workload (without lists, the
    call's other launch configuration) against the oracle's stored cores; and
    a sample recomputed by the oracle here, which ties the stored file to the
    oracle as it stands."""
    h = H()
    X, task = workloads.workload("hdbscan_200k_d61")
    ms = task["min_samples"]
    core = np_(h.core_distances(dev(X), ms, lists=False))
    oc = golden_outputs("hdbscan_200k_d61", X)["core"]
    parity.check_core(core, oc, where="200k, every core")
    rng = np.random.default_rng(1)
    rows = np.sort(rng.choice(X.shape[1], 300, replace=False))
    assert np.array_equal(oracle.core_distances(X, ms, rows=rows), oc[rows])
