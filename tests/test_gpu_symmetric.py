"""The symmetric Boruvka scan (each unordered pair once, per-component bounds,
recorded pairs weighed exactly) against the one-sided scan and the FP32
FFMA engine: the same tree bit for bit, and against the oracle's tree where
the oracle is cheap.  The symmetric form is forced in every round here;
by default it runs only where at least half the points need a scan."""

import numpy as np
import pytest

import goldens
import oracle
import oracle_pins
import parity
import workloads
from gpu_common import H, dev, np_

pytestmark = pytest.mark.gpu


@pytest.fixture
def h():
    mod = H()
    pe = mod.set_engine("auto")
    pf = mod.set_scan_form("auto")
    pp = mod.set_scan_pruning(True)
    yield mod
    mod.set_engine(pe)
    mod.set_scan_form(pf)
    mod.set_scan_pruning(pp)


def tree(h, X, ms, engine="auto", form="auto", shortcuts=True, prune=True, pairs=False):
    h.set_engine(engine)
    h.set_scan_form(form)
    h.set_scan_pruning(prune)
    Xd = dev(X)
    core, idx, dist = h.core_distances(Xd, ms)
    if shortcuts:
        e, w = h.mr_mst(Xd, core, idx, dist)
    else:
        e, w = h.mr_mst(Xd, core)
    e = np_(e)
    rec = h.last_mst_symmetric()
    scanned = h.last_mst_scan_pairs()
    h.set_engine("auto")
    h.set_scan_form("auto")
    h.set_scan_pruning(True)
    out = (e[:, 0].astype(np.int64), e[:, 1].astype(np.int64), np_(w), rec)
    return out + (scanned,) if pairs else out


def same(a, b):
    return all(np.array_equal(u, v) for u, v in zip(a[:3], b[:3]))


@pytest.mark.parametrize("n,d,ms", [(200, 61, 3), (1000, 61, 10), (1000, 64, 5), (777, 33, 7),
                                    (1500, 32, 4), (2000, 17, 10), (3000, 48, 1), (129, 8, 2)])
def test_symmetric_matches_one_sided_and_simt(h, n, d, ms):
    """Ragged sizes, 8 to 64 features (TF32 operands up to 32, FP16 above):
    the three scans build the same tree, and it is the oracle's."""
    X = workloads.small(n, d, seed=n + 31 * d, dup_frac=0.03, outlier_frac=0.08)
    s = tree(h, X, ms, form="symmetric")
    o = tree(h, X, ms, form="one_sided")
    f = tree(h, X, ms, engine="simt")
    assert same(s, o) and same(s, f)
    assert any(r >= 0 for r in s[3]), s[3]  # some round ran symmetric
    assert all(r == -1 for r in o[3])
    oc = oracle.core_distances(X, ms)
    olo, ohi, ow = oracle.prim_mst(X, oc)
    floor = 1e-5 * float(np.median(oc))
    parity.check_mst(n, s[0], s[1], s[2], olo, ohi, ow,
                     lambda a, b: oracle.mr_weights(X, oc, a, b), floor, where=f"sym n={n} d={d}")


@pytest.mark.parametrize("g", goldens.all_fixtures(), ids=lambda g: g["name"])
def test_symmetric_golden(h, g):
    """Hand-worked trees with exact ties: the edges must be exactly those."""
    lo, hi, w, _ = tree(h, g["X"], g["min_samples"], form="symmetric")
    assert [(int(a), int(b)) for a, b in zip(lo, hi)] == [(a, b) for a, b, _ in g["edges"]]
    assert np.allclose(w, [c for _, _, c in g["edges"]], rtol=1e-6, atol=0)


@pytest.mark.parametrize("seed,n,d,ms", [(1, 200, 2, 3), (2, 500, 3, 5), (3, 1000, 4, 10),
                                         (5, 700, 6, 1), (6, 3000, 5, 4), (4, 130, 1, 2),
                                         (7, 3000, 1, 2)])
def test_symmetric_integer_ties(h, seed, n, d, ms):
    """Integer coordinates with many equal weights: ties by (w, lo, hi) decide
    the tree, which must be the oracle's edge for edge.  In one dimension most
    points have copies, so many bounds are exactly 0 (the filter must still
    pass equal weights)."""
    rng = np.random.default_rng(seed)
    X = oracle_pins.int_points(rng, n, d, span=3, dup_frac=0.2)
    lo, hi, w, _ = tree(h, X, ms, form="symmetric")
    oc = oracle.core_distances(X, ms)
    olo, ohi, ow = oracle.prim_mst(X, oc)
    assert np.array_equal(lo, olo) and np.array_equal(hi, ohi)
    assert np.array_equal(w.astype(np.float64), ow.astype(np.float32).astype(np.float64))


def test_symmetric_50k(h):
    """The 50k-clip workload: symmetric, one-sided and FP32 trees identical,
    and few pairs recorded (the bounds tighten quickly)."""
    X, task = workloads.workload("hdbscan_50k_d61")
    ms = task["min_samples"]
    s = tree(h, X, ms, form="symmetric")
    o = tree(h, X, ms, form="one_sided")
    f = tree(h, X, ms, engine="simt")
    assert same(s, o) and same(s, f)
    n = X.shape[1]
    assert all(0 <= r <= 20 * n for r in s[3]), s[3]


def test_symmetric_default_200k_rounds(h):
    """The 200k-clip workload under the default form: the late rounds, where
    most points need a scan, run symmetric; the tree equals the one-sided
    scan's."""
    X, task = workloads.workload("hdbscan_200k_d61")
    ms = task["min_samples"]
    a = tree(h, X, ms)
    o = tree(h, X, ms, form="one_sided")
    assert same(a, o)
    assert any(r >= 0 for r in a[3]) and any(r == -1 for r in a[3]), a[3]


def test_symmetric_wide_dynamic_range(h):
    """A few points 1e5 away from unit-scale clusters: the FP16 form's
    absolute error is large against the clusters' distances, so many pairs
    are recorded; the tree stays the FP32 engine's."""
    X = workloads.small(20000, 48, seed=21, dup_frac=0.01).astype(np.float64)
    X /= np.abs(X).max()
    X[:, :8] *= 1.0e5
    X = np.ascontiguousarray(X, dtype=np.float32)
    s = tree(h, X, 7, form="symmetric")
    f = tree(h, X, 7, engine="simt")
    assert same(s, f)


def test_symmetric_without_lists_is_one_sided(h):
    """Without nearest lists there is no bound: the scan stays one-sided."""
    X = workloads.small(1000, 40, seed=5)
    s = tree(h, X, 5, form="symmetric", shortcuts=False)
    assert all(r == -1 for r in s[3])
    f = tree(h, X, 5, engine="simt", shortcuts=False)
    assert same(s, f)


def test_symmetric_far_from_origin(h):
    """Norms far above the distances: the bound's conversion works near its
    rounding limit."""
    X = workloads.small(5000, 40, seed=8, dup_frac=0.02) + np.float32(300.0)
    X = np.ascontiguousarray(X, dtype=np.float32)
    s = tree(h, X, 5, form="symmetric")
    f = tree(h, X, 5, engine="simt")
    assert same(s, f)


def mixture(n, d, seed, clusters=20, outlier_frac=0.05, dup_frac=0.0, mean_sd=4.0):
    return workloads.draw(workloads.Mixture(n=n, d=d, clusters=clusters, mean_sd=mean_sd,
                                            sigma=None, sigma_range=(0.5, 2.0),
                                            outlier_frac=outlier_frac, dup_frac=dup_frac,
                                            seed=seed))


def pruned_vs_unpruned(h, X, ms):
    a = tree(h, X, ms, form="symmetric", pairs=True)
    b = tree(h, X, ms, form="symmetric", prune=False, pairs=True)
    o = tree(h, X, ms, form="one_sided")
    assert same(a, b) and same(a, o)
    return a, b


def test_pruned_50k(h):
    """The 50k-clip workload (block pruning on: at least 16 384 points): the
    pruned, unpruned and one-sided scans give the same tree, and the
    pruned one evaluates fewer pairs."""
    X, task = workloads.workload("hdbscan_50k_d61")
    a, b = pruned_vs_unpruned(h, X, task["min_samples"])
    assert a[4] < b[4], (a[4], b[4])


@pytest.mark.parametrize("n,d,ms,seed", [(20000, 40, 7, 1), (30000, 64, 10, 2), (16384, 33, 5, 3),
                                         (17001, 20, 4, 4)])
def test_pruned_mixtures(h, n, d, ms, seed):
    """Clustered sets with outliers, ragged block counts, 20 to 64 features."""
    X = mixture(n, d, seed=seed)
    pruned_vs_unpruned(h, X, ms)


def test_pruned_heavy_duplicates(h):
    """Every point has many exact copies: equal weights everywhere, decided by
    the index order."""
    rng = np.random.default_rng(4)
    base = mixture(400, 24, seed=5, outlier_frac=0.0)
    X = np.ascontiguousarray(base[:, rng.integers(0, 400, size=24000)])
    pruned_vs_unpruned(h, X, 6)


def test_pruned_far_from_origin(h):
    """Norms far above the distances."""
    X = np.ascontiguousarray(mixture(20000, 32, seed=11) + np.float32(300.0), dtype=np.float32)
    pruned_vs_unpruned(h, X, 7)


def test_pruned_many_small_clusters(h):
    """Hundreds of small clusters: more components than the grouping takes in
    the early rounds (those run unpruned), fewer later."""
    X = mixture(40000, 16, seed=9, clusters=600, outlier_frac=0.02, mean_sd=6.0)
    pruned_vs_unpruned(h, X, 5)


def test_list_overflow_falls_back(h):
    """Lists capped at 3 pairs: the symmetric rounds that record more
    overflow and are redone one-sided, and the open rows' rescan overflows to
    the FP32 exact scan; the tree stays the one-sided FP32 tree."""
    X = mixture(20000, 40, seed=13, dup_frac=0.02)
    f = tree(h, X, 7, engine="simt")
    prev = h.set_scan_list_cap(3)
    try:
        s = tree(h, X, 7, form="symmetric")
        o = tree(h, X, 7, form="one_sided")
    finally:
        h.set_scan_list_cap(prev)
    assert same(s, f) and same(o, f)
    assert -1 in s[3] and all(r <= 3 for r in s[3]), s[3]  # overflowing rounds fell back
