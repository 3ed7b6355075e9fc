"""Checks that pin the oracle to something other than itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises ``AssertionError``
on the first disagreement.  The references are:

* hand-worked fixtures (``tests/golden``), from the definitions on page
  "HDBSCAN" (gpu/hdbscan), "The algorithm on the device";
* a second MST algorithm written here (Kruskal over every pair, union-find),
  on integer coordinates where every weight is exact in float64;
* scipy's minimum spanning tree, to which the method reduces when
  min_samples = 1 (every core distance is 0, so the weight is the distance);
* brute-force k-NN by numpy sorting of every distance, integer coordinates;
* invariants of any MST (cut and cycle properties, n - 1 edges, a tree) and of
  core distances (non-decreasing in min_samples, 0 at min_samples = 1).

``tests/test_oracle.py`` runs them on the oracle, and also on deliberately
broken copies of it to show each planted mistake fails at least one pin.
"""

from __future__ import annotations

import math

import numpy as np

import goldens


# ---------------------------------------------------------------------------
# independent helpers (numpy; none calls the oracle)

def np_dist(X) -> np.ndarray:
    """Dense float64 distance matrix of the columns of X [d, n]."""
    P = np.asarray(X, dtype=np.float64).T
    sq = ((P[:, None, :] - P[None, :, :]) ** 2).sum(axis=2)
    return np.sqrt(sq)


def np_knn(X, Y, k):
    Q = np.asarray(X, dtype=np.float64).T
    P = np.asarray(Y, dtype=np.float64).T
    D = np.sqrt(((Q[:, None, :] - P[None, :, :]) ** 2).sum(axis=2))
    idx = np.empty((Q.shape[0], k), dtype=np.int64)
    for i in range(Q.shape[0]):
        order = np.lexsort((np.arange(P.shape[0]), D[i]))  # by distance, then index
        idx[i] = order[:k]
    return idx, np.take_along_axis(D, idx, axis=1)


def np_core(X, ms):
    D = np_dist(X)
    return np.sort(D, axis=1)[:, ms - 1]


class DSU:
    def __init__(self, n):
        self.p = list(range(n))

    def find(self, x):
        while self.p[x] != x:
            self.p[x] = self.p[self.p[x]]
            x = self.p[x]
        return x

    def union(self, a, b):
        ra, rb = self.find(a), self.find(b)
        if ra == rb:
            return False
        self.p[ra] = rb
        return True


def kruskal(W):
    """MST of the dense weight matrix W by Kruskal under (w, lo, hi)."""
    n = W.shape[0]
    lo, hi = np.triu_indices(n, 1)
    w = W[lo, hi]
    order = np.lexsort((hi, lo, w))
    dsu = DSU(n)
    out = []
    for e in order:
        if dsu.union(int(lo[e]), int(hi[e])):
            out.append((int(lo[e]), int(hi[e]), float(w[e])))
            if len(out) == n - 1:
                break
    return out


def is_spanning_tree(n, lo, hi):
    if len(lo) != n - 1:
        return False
    dsu = DSU(n)
    return all(dsu.union(int(a), int(b)) for a, b in zip(lo, hi))


def int_points(rng, n, d, span=4, dup_frac=0.2):
    """Small integer coordinates: every squared distance is an exact float64
    integer, so any summation order gives the same bits; many exact ties."""
    P = rng.integers(-span, span + 1, size=(n, d)).astype(np.float32)
    nd = int(dup_frac * n)
    if nd:
        t = rng.choice(n, size=nd, replace=False)
        s = rng.integers(0, n, size=nd)
        P[t] = P[s]
    return np.ascontiguousarray(P.T)


# ---------------------------------------------------------------------------
# pins

def pin_golden(o):
    for g in goldens.all_fixtures():
        X, ms = g["X"], g["min_samples"]
        core = o.core_distances(X, ms)
        assert np.allclose(core, g["core"], rtol=1e-12, atol=1e-12), (g["name"], core, g["core"])
        if g["knn"]:
            idx, dist = o.knn(X, X, g["knn_k"])
            assert (idx == np.array(g["knn"])).all(), (g["name"], idx)
            assert np.allclose(dist, np.array(g["knn_dist"]), rtol=1e-12, atol=0), (g["name"], dist)
        lo, hi, w = o.prim_mst(X, core)
        exp = g["edges"]
        assert [(int(a), int(b)) for a, b in zip(lo, hi)] == [(a, b) for a, b, _ in exp], (
            g["name"], list(zip(lo, hi)))
        assert np.allclose(w, [c for _, _, c in exp], rtol=1e-12, atol=1e-12), (g["name"], w)
        assert math.isclose(w.sum(), g["total"], rel_tol=1e-12, abs_tol=1e-12), (g["name"], w.sum())


def pin_kruskal(o, seeds=(1, 2, 3, 4), sizes=((7, 1), (40, 2), (120, 3), (200, 5))):
    """Prim (oracle) and Kruskal (here) give the same edges on exact weights."""
    for seed in seeds:
        rng = np.random.default_rng(seed)
        for n, d in sizes:
            X = int_points(rng, n, d)
            for ms in (1, 2, 4):
                core = np_core(X, ms)
                oc = o.core_distances(X, ms)
                assert np.array_equal(oc, core), ("core", seed, n, ms)
                W = np.maximum(np_dist(X), np.maximum(core[:, None], core[None, :]))
                ref = kruskal(W)
                lo, hi, w = o.prim_mst(X, oc)
                got = [(int(a), int(b), float(c)) for a, b, c in zip(lo, hi, w)]
                assert got == ref, ("kruskal", seed, n, d, ms)


def pin_scipy_emst(o):
    """min_samples = 1 gives core 0 and the Euclidean MST: total weight equals scipy's."""
    from scipy.sparse.csgraph import minimum_spanning_tree
    rng = np.random.default_rng(7)
    for n, d in ((30, 2), (300, 5), (800, 61)):
        X = rng.normal(size=(d, n)).astype(np.float32)
        core = o.core_distances(X, 1)
        assert np.array_equal(core, np.zeros(n)), "core at min_samples 1"
        lo, hi, w = o.prim_mst(X, core)
        ref = minimum_spanning_tree(np_dist(X)).sum()
        assert math.isclose(w.sum(), ref, rel_tol=1e-12), ("emst", n, d, w.sum(), ref)


def pin_bruteforce_knn(o):
    rng = np.random.default_rng(11)
    for n, m, d, k in ((50, 50, 1, 7), (120, 90, 3, 10), (200, 200, 2, 16), (17, 5, 4, 5)):
        X = int_points(rng, n, d)
        Y = int_points(rng, m, d)
        for A, B in ((X, Y), (X, X)):
            kk = min(k, B.shape[1])
            ri, rd = np_knn(A, B, kk)
            oi, od = o.knn(A, B, kk)
            assert np.array_equal(oi, ri), ("knn idx", n, m, d, k)
            assert np.array_equal(od, rd), ("knn dist", n, m, d, k)


def pin_invariants(o):
    # integer coordinates: the numpy weights below are then bit-identical to any
    # correct float64 evaluation, so the cut and cycle checks see the same ties
    rng = np.random.default_rng(5)
    for n, d, ms, dup, span in ((150, 4, 3, 0.0, 30), (200, 8, 5, 0.1, 6), (90, 61, 2, 0.05, 3)):
        X = int_points(rng, n, d, span=span, dup_frac=dup)
        cores = [o.core_distances(X, s) for s in range(1, ms + 2)]
        for a, b in zip(cores, cores[1:]):
            assert (b >= a).all(), "core must not decrease with min_samples"
        assert (cores[0] == 0).all(), "core at min_samples 1 is 0"
        core = cores[ms - 1]
        idx, dist = o.knn(X, X, min(12, n))
        assert (np.diff(dist, axis=1) >= 0).all(), "k-NN distances sorted"
        lo, hi, w = o.prim_mst(X, core)
        assert (lo < hi).all(), "lo < hi"
        assert is_spanning_tree(n, lo, hi), "n - 1 edges forming a tree"
        D = np_dist(X)
        W = np.maximum(D, np.maximum(core[:, None], core[None, :]))
        assert np.allclose(w, W[lo, hi], rtol=1e-12, atol=1e-12), "edge weights"
        assert (w >= np.maximum(core[lo], core[hi])).all()
        keys = list(zip(w, lo, hi))
        assert keys == sorted(keys), "edges sorted by (w, lo, hi)"
        in_tree = set(zip(lo.tolist(), hi.tolist()))
        # cut property: the least crossing edge of a random cut is a tree edge
        for _ in range(100):
            S = rng.random(n) < rng.uniform(0.05, 0.95)
            if S.all() or not S.any():
                continue
            a, b = np.nonzero(S[:, None] & ~S[None, :])
            la, hb = np.minimum(a, b), np.maximum(a, b)
            e = np.lexsort((hb, la, W[a, b]))[0]
            assert (int(la[e]), int(hb[e])) in in_tree, "cut property"
        # cycle property: every non-tree edge is the heaviest on its tree cycle
        adj = [[] for _ in range(n)]
        for a, b, c in zip(lo, hi, w):
            adj[a].append((b, (c, a, b)))
            adj[b].append((a, (c, a, b)))
        for s in range(0, n, max(1, n // 40)):
            best = {s: (-1.0, -1, -1)}
            stack = [s]
            while stack:
                u = stack.pop()
                for v, key in adj[u]:
                    if v not in best:
                        best[v] = max(best[u], key)
                        stack.append(v)
            for t in range(n):
                if t == s or (min(s, t), max(s, t)) in in_tree:
                    continue
                key = (W[s, t], min(s, t), max(s, t))
                assert key > best[t], "cycle property"


ALL_PINS = (pin_golden, pin_kruskal, pin_scipy_emst, pin_bruteforce_knn, pin_invariants)


# ---------------------------------------------------------------------------
# pins of the back half (oracle/hierarchy.py): labels from the spanning tree

def _partition_equal(a, b):
    """Same clusters and same noise, up to the numbering of the clusters."""
    a = np.asarray(a)
    b = np.asarray(b)
    if a.shape != b.shape or not np.array_equal(a < 0, b < 0):
        return False
    pairs = set(zip(a[a >= 0].tolist(), b[b >= 0].tolist()))
    return (len(pairs) == len(set(p[0] for p in pairs)) == len(set(p[1] for p in pairs)))


def pin_hierarchy_golden(o, h):
    """Hand-worked labels (tests/golden, the fixtures with a labels line)."""
    for g in goldens.all_fixtures():
        if "labels" not in g:
            continue
        core = o.core_distances(g["X"], g["min_samples"])
        lo, hi, w = o.prim_mst(g["X"], core)
        got = h.hdbscan_labels(g["X"].shape[1], lo, hi, w, g["min_cluster_size"])
        assert np.array_equal(got, g["labels"]), (g["name"], got, g["labels"])


def pin_hierarchy_sklearn(o, h):
    """scikit-learn's HDBSCAN (the page's upstream) on random blobs.

    With min_samples = 1 every weight is a distinct distance, the spanning tree
    is unique, and the partitions must be equal.  With min_samples > 1 most
    points join the tree at exactly their core distance, often through one of
    several equal edges, and the two programs may place such a point in a
    cluster or in noise differently (page "HDBSCAN", "A lesson about tests:
    ties"): there, after matching each cluster to the one it overlaps most, at
    most 3% of the points may disagree."""
    try:
        from sklearn.cluster import HDBSCAN
    except ImportError:  # pragma: no cover - not installed on every machine
        return
    rng = np.random.default_rng(17)
    for n, d, k, ms, mcs in ((300, 2, 4, 1, 10), (250, 3, 3, 1, 5), (600, 8, 6, 1, 20),
                             (300, 2, 4, 5, 10), (600, 8, 6, 10, 20), (400, 61, 5, 3, 15)):
        means = rng.normal(0.0, 6.0, size=(k, d))
        lab = rng.integers(0, k, size=n)
        P = (means[lab] + rng.normal(size=(n, d)) * rng.uniform(0.5, 2.0, size=(k, 1))[lab])
        P[: n // 20] = rng.uniform(P.min(0), P.max(0), size=(n // 20, d))
        X = np.ascontiguousarray(P.astype(np.float32).T)
        core = o.core_distances(X, ms)
        lo, hi, w = o.prim_mst(X, core)
        got = h.hdbscan_labels(n, lo, hi, w, mcs)
        ref = HDBSCAN(min_cluster_size=mcs, min_samples=ms, copy=True).fit(
            X.T.astype(np.float64)).labels_
        if ms == 1:
            assert _partition_equal(got, ref), ("sklearn", n, d, ms, mcs)
            continue
        assert len(set(got.tolist())) == len(set(ref.tolist())), ("cluster count", n, ms)
        mapped = np.full(n, -1)
        for c in set(got.tolist()) - {-1}:
            vals, cnt = np.unique(ref[got == c], return_counts=True)
            mapped[got == c] = vals[np.argmax(cnt)]
        assert np.mean(mapped != ref) <= 0.03, ("sklearn", n, d, ms, mcs, np.mean(mapped != ref))


def pin_hierarchy_invariants(o, h):
    """Every cluster holds at least min_cluster_size points; clusters are
    numbered by first appearance; an isolated far point is noise; a single
    blob of exactly min_cluster_size points has no cluster (the root is never
    selected)."""
    rng = np.random.default_rng(23)
    for n, d, ms, mcs in ((500, 4, 5, 12), (300, 2, 2, 6), (120, 6, 4, 30)):
        P = rng.normal(size=(n, d)) * 0.3 + rng.integers(0, 4, size=(n, 1)) * 5.0
        X = np.ascontiguousarray(P.astype(np.float32).T)
        core = o.core_distances(X, ms)
        lo, hi, w = o.prim_mst(X, core)
        lab = h.hdbscan_labels(n, lo, hi, w, mcs)
        ids = [v for v in lab.tolist() if v >= 0]
        first = []
        for v in ids:
            if v not in first:
                first.append(v)
        assert first == list(range(len(first))), "numbering by first appearance"
        for c in set(ids):
            assert ids.count(c) >= mcs, "cluster below min_cluster_size"
    X = np.array([[0.0, 0.1, 0.2, 0.3, 0.4, 100.0]], dtype=np.float32)
    core = o.core_distances(X, 2)
    lo, hi, w = o.prim_mst(X, core)
    assert h.hdbscan_labels(6, lo, hi, w, 5).tolist() == [-1] * 6, "one blob: no cluster"
    assert h.hdbscan_labels(6, lo, hi, w, 2)[5] == -1, "a far point is noise"


HIERARCHY_PINS = (pin_hierarchy_golden, pin_hierarchy_sklearn, pin_hierarchy_invariants)
