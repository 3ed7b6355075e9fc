"""Exact k-NN on the GPU against the float64 oracle (parity rules in parity.py)."""

import numpy as np
import pytest

import oracle
import oracle_pins
import parity
import workloads
from gpu_common import H, dev, golden_outputs, np_, oracle_knn_check

pytestmark = pytest.mark.gpu

# ragged sizes: single points, below / across / past one 128-wide tile, several tiles
CASES = [
    # n, m, d, k
    (1, 1, 1, 1), (2, 3, 1, 2), (3, 5, 3, 5), (5, 2, 61, 1), (127, 129, 61, 10),
    (129, 127, 64, 10), (130, 300, 65, 7), (1001, 777, 102, 10), (2000, 400, 192, 16),
    (300, 2000, 3, 12), (257, 1000, 61, 13), (600, 640, 61, 32), (40, 40, 17, 32),
    # past the tensor tile's 192 features: rows padded to 208 (a 16-feature
    # last segment in the refine) and to 256
    (300, 400, 200, 10), (129, 257, 250, 16),
]


@pytest.mark.parametrize("n,m,d,k", CASES)
def test_knn_ragged(n, m, d, k):
    h = H()
    X = workloads.small(n, d, seed=n * 7 + d, dup_frac=0.05)
    Y = workloads.small(m, d, seed=m * 11 + d + 1, dup_frac=0.05)
    gi, gd = h.knn(dev(X), dev(Y), k)
    oracle_knn_check(X, Y, k, np_(gi), np_(gd), where=f"n={n} m={m} d={d} k={k}")


@pytest.mark.parametrize("n,d,k", [(1, 5, 1), (129, 61, 11), (1000, 61, 11), (777, 102, 6)])
def test_knn_self(n, d, k):
    """Y = X: every query finds itself first unless a lower-index copy exists."""
    h = H()
    X = workloads.small(n, d, seed=3 + n, dup_frac=0.1)
    Xd = dev(X)
    gi, gd = h.knn(Xd, Xd, k)
    oracle_knn_check(X, X, k, np_(gi), np_(gd), where=f"self n={n}")
    assert (np_(gd)[:, 0] == 0).all()


@pytest.mark.parametrize("seed,n,m,d,k", [(1, 300, 300, 3, 10), (2, 500, 200, 5, 16),
                                          (3, 1000, 1000, 2, 20), (4, 257, 257, 8, 32)])
def test_knn_exact_ties_integer_points(seed, n, m, d, k):
    """Integer coordinates: every distance is exact on both sides, so the index
    lists must equal the oracle's exactly, ties included (lowest index first)."""
    h = H()
    rng = np.random.default_rng(seed)
    X = oracle_pins.int_points(rng, n, d, span=3)
    Y = oracle_pins.int_points(rng, m, d, span=3)
    gi, gd = h.knn(dev(X), dev(Y), k)
    oi, od = oracle.knn(X, Y, k)
    assert np.array_equal(np_(gi), oi)
    assert np.array_equal(np_(gd).astype(np.float64), od.astype(np.float32).astype(np.float64))


def test_knn_many_copies_uses_exact_rows():
    """Blocks of 40 identical points: the expansion cannot separate the ties,
    the proof fails and the rows are searched again exactly."""
    h = H()
    base = workloads.small(50, 61, seed=5)
    X = np.ascontiguousarray(np.repeat(base, 40, axis=1))
    gi, gd = h.knn(dev(X), dev(X), 10)
    oi, od = oracle.knn(X, X, 10)
    assert np.array_equal(np_(gi), oi)


def test_knn_strided_input():
    h = H()
    import torch
    X = workloads.small(500, 61, seed=8)
    big = torch.zeros((61, 700), dtype=torch.float32, device="cuda")
    big[:, :500] = dev(X)
    view = big[:, :500]
    assert view.stride(0) == 700
    gi, gd = h.knn(view, view, 10)
    oracle_knn_check(X, X, 10, np_(gi), np_(gd), where="strided")


def test_knn_host_inputs_round_trip():
    h = H()
    X = workloads.small(200, 20, seed=4)
    gi, gd = h.knn(X, X, 5)
    assert not gi.is_cuda
    oracle_knn_check(X, X, 5, gi.numpy(), gd.numpy(), where="host")


def test_knn_nonfinite_rejected():
    h = H()
    X = workloads.small(100, 8, seed=2)
    X[3, 17] = np.nan
    with pytest.raises(h.HdbmstError) as e:
        h.knn(dev(X), dev(X), 4)
    assert e.value.status == 4


def test_knn_bad_k():
    h = H()
    X = workloads.small(10, 4, seed=2)
    with pytest.raises(h.HdbmstError):
        h.knn(dev(X), dev(X), 11)
    with pytest.raises(h.HdbmstError):
        h.knn(dev(X), dev(workloads.small(40, 4, seed=3)), 33)


def test_knn_section_1416_d102():
    """Kilosort4-style section: 1 416 x 102, k = 10 against every 5th point; all rows."""
    h = H()
    X, task = workloads.workload("knn_1416_d102")
    Y = workloads.subset_columns(X, task["y_stride"])
    assert Y.shape == (102, 284)
    gi, gd = h.knn(dev(X), dev(Y), task["k"])
    oracle_knn_check(X, Y, task["k"], np_(gi), np_(gd), where="1416x102")


def test_knn_200k_d192():
    """200 000 x 192 against 20 000 (every 10th point), k = 10, in the
    benchmark's launch configuration: every row against the oracle's k + 1
    nearest (stored by make_oracle_totals.py from the oracle alone; their
    distances recomputed here by the oracle's pair distance, the same float64
    terms in the same order), by the gap-aware parity rules."""
    h = H()
    X, task = workloads.workload("knn_200k_d192")
    Y = workloads.subset_columns(X, task["y_stride"])
    k = task["k"]
    gi, gd = h.knn(dev(X), dev(Y), k)
    gi, gd = np_(gi), np_(gd)
    n, m = X.shape[1], Y.shape[1]
    g = golden_outputs("knn_200k_d192", X)
    assert int(g["k"]) == k
    oi = g["idx"].astype(np.int64)
    assert oi.shape == (n, k + 1)
    od = oracle.pair_dist_xy(X, Y, np.repeat(np.arange(n), k + 1), oi.ravel()).reshape(n, k + 1)
    dd, ii = np.diff(od, axis=1), np.diff(oi, axis=1)
    assert ((dd > 0) | ((dd == 0) & (ii > 0))).all(), "stored lists out of (dist, idx) order"
    # the subset holds every 10th query itself: those rows find themselves at 0
    selfrows = np.arange(0, n, 10)
    assert (gd[selfrows, 0] == 0).all()

    def pd(r, c):
        return oracle.pair_dist_xy(X, Y, r, c)

    parity.check_knn(gi, gd, oi, od, k, m, pd, where="200k x 192, all rows")
