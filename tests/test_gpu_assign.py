"""Bipartite modularity assignment on the GPU against the oracle
(oracle/bipartite.py; page "Kilosort4 clustering and matching", section
"Assignment in parallel: why the graph is bipartite").

Labels are integers decided by float64 scores that both sides evaluate with
the same operations, so the labels, the number of rounds and the spikes moved
per round must be identical.  The graphs are the oracle's own k-NN lists (no
input comes from the CUDA path); the initial subset labels are seeded draws
(the page seeds them by k-means++, which is outside this path).
"""

import numpy as np
import pytest

import oracle
from oracle import bipartite as B
import workloads
from gpu_common import H, dev, golden_outputs, np_

pytestmark = pytest.mark.gpu


def run_both(h, nbr, m, right0, C, gamma, max_rounds=200):
    gl, gr, grounds, gmoved = h.bipartite_assign(dev(np.asarray(nbr, dtype=np.int32)), m,
                                                 dev(np.asarray(right0, dtype=np.int32)), C,
                                                 gamma, max_rounds)
    ol, orr, orounds, omoved = B.assign(nbr, m, right0, C, gamma, max_rounds)
    assert np.array_equal(np_(gl), ol), "left labels"
    assert np.array_equal(np_(gr), orr), "right labels"
    assert grounds == orounds and gmoved == omoved, (grounds, orounds, gmoved, omoved)
    return ol, orr, orounds


def test_hand_graphs():
    h = H()
    run_both(h, np.array([[0, 1]] * 3 + [[2, 3]] * 3), 4, [0, 0, 1, 1], 2, 1.0)
    nbr_c = np.array([[0, 1, 2], [0, 1, 3], [0, 1, 3], [0, 1, 3]])
    l, r, _ = run_both(h, nbr_c, 4, [0, 0, 1, 0], 2, 1.0)
    assert l.tolist() == [1, 0, 0, 0]
    l, r, _ = run_both(h, nbr_c, 4, [0, 0, 1, 0], 2, 0.5)
    assert l.tolist() == [0, 0, 0, 0]
    run_both(h, np.array([[0, 1], [1, 2], [1, 2]]), 3, [3, 1, 1], 4, 0.0)
    run_both(h, np.array([[0, 1]] * 3), 2, [0, 0], 2, 3.0)
    run_both(h, np.array([[0, 1], [0, 1]]), 3, [2, 2, 1], 3, 1.0)


@pytest.mark.parametrize("n, m, k, C, gamma", [
    (1, 1, 1, 1, 1.0), (37, 11, 3, 5, 1.0), (300, 64, 10, 20, 0.0), (300, 64, 10, 20, 0.3),
    (1000, 200, 10, 200, 1.0), (257, 300, 32, 7, 2.0), (500, 40, 17, 3, 0.5),
    (2000, 5000, 10, 300, 1.0),
])
def test_random_graphs(n, m, k, C, gamma):
    h = H()
    rng = np.random.default_rng(n + 7 * m + k)
    nbr = np.stack([rng.choice(m, k, replace=False) for _ in range(n)])
    right0 = rng.integers(0, C, m)
    run_both(h, nbr, m, right0, C, gamma)


def test_round_cap_and_empty():
    h = H()
    rng = np.random.default_rng(5)
    nbr = np.stack([rng.choice(50, 6, replace=False) for _ in range(400)])
    right0 = rng.integers(0, 30, 50)
    _, _, rounds = run_both(h, nbr, 50, right0, 30, 1.0, max_rounds=1)
    assert rounds == 1
    gl, gr, rounds, moved = h.bipartite_assign(dev(np.zeros((0, 4), dtype=np.int32)), 5,
                                               dev(np.array([1, 0, 2, 2, 1], dtype=np.int32)), 3)
    assert gl.shape == (0,) and np_(gr).tolist() == [1, 0, 2, 2, 1] and moved == [0]


def test_bad_inputs_rejected():
    h = H()
    good = np.array([[0, 1], [1, 2]], dtype=np.int32)
    with pytest.raises(h.HdbmstError) as e:
        h.bipartite_assign(dev(np.array([[0, 3], [1, 2]], dtype=np.int32)), 3,
                           dev(np.array([0, 0, 0], dtype=np.int32)), 2)
    assert e.value.status == 1
    with pytest.raises(h.HdbmstError) as e:
        h.bipartite_assign(dev(good), 3, dev(np.array([0, 5, 0], dtype=np.int32)), 2)
    assert e.value.status == 1
    with pytest.raises(h.HdbmstError) as e:
        h.bipartite_assign(dev(good), 3, dev(np.array([0, 1, 0], dtype=np.int32)), 2, gamma=-1.0)
    assert e.value.status == 1


def test_section_1416_d102():
    """The Kilosort4-style section: the oracle's k = 10 lists of 1 416 spikes
    against every 5th point, 200 initial clusters (the page's seed count)."""
    h = H()
    X, task = workloads.workload("knn_1416_d102")
    Y = workloads.subset_columns(X, task["y_stride"])
    oi, _ = oracle.knn(X, Y, task["k"])
    rng = np.random.default_rng(11)
    right0 = rng.integers(0, 200, Y.shape[1])
    for gamma in (0.5, 1.0):
        _, _, rounds = run_both(h, oi, Y.shape[1], right0, 200, gamma)
        assert rounds < 200
    # the whole path on the GPU: its k-NN lists equal the oracle's here, and
    # the assignment on them is the oracle's
    gi, _ = h.knn(dev(X), dev(Y), task["k"])
    assert np.array_equal(np_(gi), oi)


def test_knn_200k_d192_graph():
    """200 000 spikes, k = 10 against the 20 000-point subset: the oracle's
    stored lists (their first k entries), 200 initial clusters."""
    h = H()
    X, task = workloads.workload("knn_200k_d192")
    k = task["k"]
    nbr = golden_outputs("knn_200k_d192", X)["idx"][:, :k].astype(np.int64)
    m = X.shape[1] // task["y_stride"]
    rng = np.random.default_rng(12)
    right0 = rng.integers(0, 200, m)
    _, _, rounds = run_both(h, nbr, m, right0, 200, 1.0)
    assert rounds < 200
