"""The tensor-core and FP32 FFMA distance tiles give bit-identical results:
both only rank candidates, every reported value is re-evaluated with the
exact distance, and each engine proves its kept set against its own rounding
bound.  Also checks the tensor-core engine against the oracle directly."""

import numpy as np
import pytest

import oracle_pins
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
    h.set_engine("simt")
    a = fn()
    h.set_engine("tensor")
    b = fn()
    h.set_engine("auto")
    return a, b


@pytest.mark.parametrize("n,m,d,k", [(1, 1, 1, 1), (5, 7, 3, 4), (129, 300, 17, 10),
                                     (1000, 1000, 61, 11), (777, 2049, 64, 16),
                                     (300, 130, 33, 32), (2000, 1500, 48, 12),
                                     # wide rows: A lo parts in shared memory
                                     (500, 700, 65, 10), (300, 1000, 102, 10),
                                     (257, 900, 192, 16), (200, 300, 150, 32)])
def test_knn_engines_identical(h, n, m, d, k):
    X = workloads.small(n, d, seed=n + 3 * d, dup_frac=0.05)
    Y = workloads.small(m, d, seed=m + 5 * d, dup_frac=0.05)
    (ai, ad), (bi, bd) = both(h, lambda: tuple(np_(t) for t in h.knn(dev(X), dev(Y), k)))
    assert np.array_equal(ai, bi) and np.array_equal(ad, bd)
    oracle_knn_check(X, Y, k, bi, bd, where=f"tensor n={n} m={m} d={d}")


def test_core_engines_identical_2k(h):
    X, task = workloads.workload("hdbscan_2k_d61")
    ms = task["min_samples"]
    a, b = both(h, lambda: tuple(np_(t) for t in h.core_distances(dev(X), ms)))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_knn_engines_integer_ties(h):
    rng = np.random.default_rng(3)
    X = oracle_pins.int_points(rng, 700, 5, span=3)
    (ai, ad), (bi, bd) = both(h, lambda: tuple(np_(t) for t in h.knn(dev(X), dev(X), 20)))
    assert np.array_equal(ai, bi) and np.array_equal(ad, bd)


def test_core_engines_identical_200k_sampled_rows(h):
    """The benchmark's workload: both engines, every row identical."""
    X, task = workloads.workload("hdbscan_200k_d61")
    ms = task["min_samples"]
    a, b = both(h, lambda: tuple(np_(t) for t in h.core_distances(dev(X), ms)))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_knn_engines_identical_200k_d192_sampled_rows(h):
    """The 200k x 192 k-NN workload (wide rows on the tensor cores): both
    engines give identical lists on every row."""
    X, task = workloads.workload("knn_200k_d192")
    Y = workloads.subset_columns(X, task["y_stride"])
    k = task["k"]
    (ai, ad), (bi, bd) = both(h, lambda: tuple(np_(t) for t in h.knn(dev(X), dev(Y), k)))
    assert np.array_equal(ai, bi) and np.array_equal(ad, bd)


@pytest.mark.parametrize("n,m,d,k", [(1000, 1000, 61, 11), (777, 2049, 64, 16), (2000, 1500, 48, 12),
                                     (300, 130, 33, 32), (20000, 20000, 61, 11),
                                     # wide rows on FP16: both A parts in TMEM
                                     (1500, 2200, 120, 10), (900, 1300, 190, 16)])
def test_fp16_tf32_simt_identical(h, n, m, d, k):
    """The two-part FP16 operands (33 to 64 features, and 97 to 128 or 161 to
    192 in the k-NN), the TF32 operands and the
    FP32 FFMA tile: identical lists; the FP16 form's ranking must be tight
    enough that the rounding proof settles almost every row (an MMA that
    computed something else would show up here as a flood of exact rows or
    as different lists)."""
    X = workloads.small(n, d, seed=n + 11 * d, dup_frac=0.02)
    Y = workloads.small(m, d, seed=m + 13 * d, dup_frac=0.02)
    out, exact = {}, {}
    for eng in ("simt", "tf32", "tensor"):
        h.set_engine(eng)
        out[eng] = tuple(np_(t) for t in h.knn(dev(X), dev(Y), k))
        exact[eng] = h.last_knn_exact_rows()
    h.set_engine("auto")
    for eng in ("tf32", "tensor"):
        assert np.array_equal(out[eng][0], out["simt"][0]), eng
        assert np.array_equal(out[eng][1], out["simt"][1]), eng
    # (k = 32 fills the whole candidate list, so every engine searches every
    # row exactly there: compare with the TF32 form's count)
    assert exact["tensor"] <= max(5, n // 100, exact["tf32"]), exact


def test_fp16_mst_identical_50k(h):
    """The Boruvka scan on the FP16 operands against the TF32 and FP32 scans:
    the same tree, bit for bit, on the 50k-clip workload."""
    X, task = workloads.workload("hdbscan_50k_d61")
    ms = task["min_samples"]
    Xd = dev(X)
    core, idx, dist = h.core_distances(Xd, ms)
    trees = {}
    for eng in ("simt", "tf32", "tensor"):
        h.set_engine(eng)
        e, w = h.mr_mst(Xd, core, idx, dist)
        trees[eng] = (np_(e), np_(w))
        if eng == "tensor":
            rounds = h.last_mst_rounds()
    h.set_engine("auto")
    for eng in ("tf32", "tensor"):
        assert np.array_equal(trees[eng][0], trees["simt"][0]), eng
        assert np.array_equal(trees[eng][1], trees["simt"][1]), eng
    scanned = sum(a for a, _, _ in rounds)
    redone = sum(x for _, _, x in rounds)
    assert redone <= max(50, scanned // 100), rounds


def test_fp16_wide_dynamic_range(h):
    """Clusters of unit scale next to a few points 1e5 away: the FP16 form's
    scale is set by the far points, its absolute error term dwarfs the
    clusters' distances, and the rounding proof must send those rows to the
    exact search rather than accept a wrong list.  Lists and trees stay
    identical to the FP32 engine's."""
    X = workloads.small(20000, 48, seed=21, dup_frac=0.01).astype(np.float64)
    X /= np.abs(X).max()
    X[:, :8] *= 1.0e5  # eight far points
    X = np.ascontiguousarray(X, dtype=np.float32)
    out, trees = {}, {}
    for eng in ("simt", "tensor"):
        h.set_engine(eng)
        out[eng] = tuple(np_(t) for t in h.core_distances(dev(X), 7))
        e, w = h.mr_mst(dev(X), *(dev(t) for t in out[eng]))
        trees[eng] = (np_(e), np_(w))
    h.set_engine("auto")
    for u, v in zip(out["simt"], out["tensor"]):
        assert np.array_equal(u, v)
    assert np.array_equal(trees["simt"][0], trees["tensor"][0])
    assert np.array_equal(trees["simt"][1], trees["tensor"][1])
