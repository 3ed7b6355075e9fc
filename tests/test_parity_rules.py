"""The parity checker itself, on the CPU: it must accept the oracle's own
answers and reject planted differences (no GPU)."""

import numpy as np
import pytest

import oracle
import oracle_pins
import parity
import workloads


def _brute_path_max(n, lo, hi, w, a, b):
    adj = [[] for _ in range(n)]
    for x, y, c in zip(lo, hi, w):
        adj[x].append((y, c))
        adj[y].append((x, c))
    best = {a: -np.inf}
    stack = [a]
    while stack:
        u = stack.pop()
        for v, c in adj[u]:
            if v not in best:
                best[v] = max(best[u], c)
                stack.append(v)
    return best[b]


def test_forest_path_max_matches_brute_force():
    X = workloads.small(60, 3, seed=3)
    core = oracle.core_distances(X, 3)
    lo, hi, w = oracle.prim_mst(X, core)
    f = parity.Forest(60, lo, hi, w)
    rng = np.random.default_rng(0)
    a = rng.integers(0, 60, 200)
    b = rng.integers(0, 60, 200)
    got = f.path_max(a, b)
    for x, y, g in zip(a, b, got):
        exp = _brute_path_max(60, lo, hi, w, x, y) if x != y else -np.inf
        assert g == exp


def _setup(n=300, d=5, ms=4):
    X = workloads.small(n, d, seed=9, dup_frac=0.05)
    core = oracle.core_distances(X, ms)
    lo, hi, w = oracle.prim_mst(X, core)
    wof = lambda a, b: oracle.mr_weights(X, core, a, b)
    return X, core, lo, hi, w, wof


def test_mst_check_accepts_oracle_tree():
    X, core, lo, hi, w, wof = _setup()
    parity.check_mst(X.shape[1], lo, hi, w.astype(np.float32), lo, hi, w, wof, 1e-5 * np.median(core))


def test_mst_check_rejects_a_swapped_edge():
    X, core, lo, hi, w, wof = _setup()
    n = X.shape[1]
    # replace the heaviest edge by another edge that reconnects the tree
    cut = int(np.argmax(w))
    keep_lo, keep_hi = np.delete(lo, cut), np.delete(hi, cut)
    f = parity.Forest(n, lo, hi, w)
    side = np.zeros(n, dtype=bool)
    # vertices on lo[cut]'s side after removing the edge
    adj = [[] for _ in range(n)]
    for a, b in zip(keep_lo, keep_hi):
        adj[a].append(b)
        adj[b].append(a)
    stack = [int(lo[cut])]
    side[lo[cut]] = True
    while stack:
        u = stack.pop()
        for v in adj[u]:
            if not side[v]:
                side[v] = True
                stack.append(v)
    a_ = np.flatnonzero(side)
    b_ = np.flatnonzero(~side)
    ww = oracle.mr_weights(X, core, np.repeat(a_, b_.size), np.tile(b_, a_.size))
    order = np.argsort(ww)
    pick = order[-1]  # the heaviest reconnecting edge: clearly not minimal
    ea, eb = int(np.repeat(a_, b_.size)[pick]), int(np.tile(b_, a_.size)[pick])
    nlo = np.append(keep_lo, min(ea, eb))
    nhi = np.append(keep_hi, max(ea, eb))
    nw = np.append(np.delete(w, cut), ww[pick])
    o = np.lexsort((nhi, nlo, nw))
    with pytest.raises(AssertionError):
        parity.check_mst(n, nlo[o], nhi[o], nw[o].astype(np.float32), lo, hi, w, wof,
                         1e-5 * np.median(core))


def test_mst_check_rejects_cycle_and_order():
    X, core, lo, hi, w, wof = _setup(n=50)
    bad_lo = lo.copy()
    bad_hi = hi.copy()
    bad_lo[-1], bad_hi[-1] = lo[0], hi[0]
    with pytest.raises(AssertionError):
        parity.check_tree_structure(50, bad_lo, bad_hi, w)
    with pytest.raises(AssertionError):
        parity.check_tree_structure(50, lo[::-1], hi[::-1], w[::-1])


def test_knn_check_accepts_oracle_and_rejects_swap():
    X = workloads.small(120, 4, seed=2, dup_frac=0.1)
    k = 6
    oi, od = oracle.knn(X, X, k + 1)
    pd = lambda r, c: oracle.pair_dist(X, r, c)
    parity.check_knn(oi[:, :k], od[:, :k].astype(np.float32), oi, od, k, 120, pd)
    gi = oi[:, :k].copy()
    gd = od[:, :k].astype(np.float32).copy()
    # put a far point in place of the nearest non-self neighbour of row 7
    far = int(np.argmax(oracle.pair_dist(X, np.full(120, 7), np.arange(120))))
    gi[7, 1] = far
    with pytest.raises(AssertionError):
        parity.check_knn(gi, gd, oi, od, k, 120, pd)


def test_core_check():
    o = np.array([0.0, 1.0, 2.0, 3.0])
    parity.check_core(o * (1 + 5e-6), o)
    with pytest.raises(AssertionError):
        parity.check_core(o * (1 + 5e-5), o)
