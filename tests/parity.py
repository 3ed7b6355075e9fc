"""Parity rules between the CUDA path and the float64 oracle.

The rules (relative tolerance ``RTOL = 1e-5``):

* k-NN, per query row, with the oracle's sorted distances ``D_0 <= D_1 <= ...``
  (the oracle lists k + 1 entries when there are more than k points):
  every oracle entry with ``D_j < D_{k-1} (1 - RTOL)`` is in the CUDA set;
  every CUDA entry lies within ``D_{k-1} (1 + RTOL)``; where the gap
  ``D_k - D_{k-1}`` exceeds ``RTOL * D_k`` the two index sets are identical;
  each CUDA distance is within RTOL of the oracle's distance for that pair;
  rows are ordered by (distance, index) and hold distinct indices.
* Core distances: ``|g - o| <= RTOL * o + RTOL * median(o)``.
* MST: ``n - 1`` edges with ``lo < hi`` forming a spanning tree, ordered by
  (w, lo, hi); each weight within RTOL (plus the core floor) of the oracle's
  float64 weight of that pair; total weight within RTOL; and every edge on one
  side only is a near-tie exchange: the heaviest edge on the other tree's path
  between its endpoints weighs the same within RTOL (the cycle property, which
  the page's tie lesson says is where Prim and Boruvka may legitimately differ:
  page "HDBSCAN", section "A lesson about tests: ties").
"""

from __future__ import annotations

import numpy as np

RTOL = 1e-5


# ---------------------------------------------------------------------------
# k-NN

def check_knn(g_idx, g_dist, o_idx, o_dist, k, m, pair_dist, rtol=RTOL, where=""):
    """``o_idx/o_dist``: oracle lists of k or k + 1 entries per row (k + 1 when m > k).
    ``pair_dist(rows, cols)``: oracle float64 distance of (row r, column j) pairs,
    row r indexing the compared rows."""
    g_idx = np.asarray(g_idx, dtype=np.int64)
    g_dist = np.asarray(g_dist, dtype=np.float64)
    nq = g_idx.shape[0]
    assert g_idx.shape == (nq, k) and g_dist.shape == (nq, k), where
    assert ((g_idx >= 0) & (g_idx < m)).all(), f"{where}: index out of range"
    # sorted by (dist, idx) with distinct indices
    for r in range(nq):
        assert len(set(g_idx[r].tolist())) == k, f"{where}: repeated index in row {r}"
    dd = np.diff(g_dist, axis=1)
    ii = np.diff(g_idx, axis=1)
    assert ((dd > 0) | ((dd == 0) & (ii > 0))).all(), f"{where}: rows not ordered by (dist, idx)"
    # oracle distance of every CUDA pair
    rows = np.repeat(np.arange(nq), k)
    o_of_g = pair_dist(rows, g_idx.ravel()).reshape(nq, k)
    err = np.abs(g_dist - o_of_g)
    bad = err > rtol * o_of_g
    assert not bad.any(), (f"{where}: distance off by more than {rtol} relative at "
                           f"{np.argwhere(bad)[:5].tolist()} (got {g_dist[bad][:5]}, "
                           f"oracle {o_of_g[bad][:5]})")
    Dk1 = o_dist[:, k - 1]
    assert (o_of_g <= Dk1[:, None] * (1 + rtol) + 0.0).all(), f"{where}: entry beyond the k-th"
    for r in range(nq):
        gs = set(g_idx[r].tolist())
        must = o_idx[r, :k][o_dist[r, :k] < Dk1[r] * (1 - rtol)]
        missing = [int(j) for j in must if int(j) not in gs]
        assert not missing, f"{where}: row {r} misses clear neighbours {missing}"
        if o_idx.shape[1] > k:
            Dk = o_dist[r, k]
            if Dk - Dk1[r] > rtol * Dk:
                assert gs == set(o_idx[r, :k].tolist()), f"{where}: row {r} set differs past a gap"


# ---------------------------------------------------------------------------
# core distances

def check_core(g, o, rtol=RTOL, where=""):
    g = np.asarray(g, dtype=np.float64)
    o = np.asarray(o, dtype=np.float64)
    floor = rtol * float(np.median(o)) if o.size else 0.0
    err = np.abs(g - o)
    bad = err > rtol * o + floor
    assert not bad.any(), (f"{where}: core off at {np.flatnonzero(bad)[:8].tolist()}: "
                           f"got {g[bad][:8]}, oracle {o[bad][:8]}")


# ---------------------------------------------------------------------------
# trees

class Forest:
    """Binary lifting over a spanning tree: heaviest edge weight on a path."""

    def __init__(self, n, lo, hi, w):
        lo = np.asarray(lo, dtype=np.int64)
        hi = np.asarray(hi, dtype=np.int64)
        w = np.asarray(w, dtype=np.float64)
        self.n = n
        adj_start = np.zeros(n + 1, dtype=np.int64)
        ends = np.concatenate([lo, hi])
        other = np.concatenate([hi, lo])
        ww = np.concatenate([w, w])
        order = np.argsort(ends, kind="stable")
        ends, other, ww = ends[order], other[order], ww[order]
        np.add.at(adj_start, ends + 1, 1)
        adj_start = np.cumsum(adj_start)
        parent = np.full(n, -1, dtype=np.int64)
        pw = np.zeros(n, dtype=np.float64)
        depth = np.zeros(n, dtype=np.int64)
        seen = np.zeros(n, dtype=bool)
        seen[0] = True
        frontier = np.array([0], dtype=np.int64)
        while frontier.size:
            nxt = []
            for u in frontier.tolist():
                for e in range(adj_start[u], adj_start[u + 1]):
                    v = other[e]
                    if not seen[v]:
                        seen[v] = True
                        parent[v] = u
                        pw[v] = ww[e]
                        depth[v] = depth[u] + 1
                        nxt.append(v)
            frontier = np.array(nxt, dtype=np.int64)
        assert seen.all(), "not a spanning tree"
        L = max(1, int(np.ceil(np.log2(max(n, 2)))) + 1)
        up = np.empty((L, n), dtype=np.int64)
        mx = np.empty((L, n), dtype=np.float64)
        up[0] = np.where(parent < 0, np.arange(n), parent)
        mx[0] = np.where(parent < 0, -np.inf, pw)
        for j in range(1, L):
            up[j] = up[j - 1][up[j - 1]]
            mx[j] = np.maximum(mx[j - 1], mx[j - 1][up[j - 1]])
        self.up, self.mx, self.depth, self.L = up, mx, depth, L

    def path_max(self, a, b):
        a = np.asarray(a, dtype=np.int64).copy()
        b = np.asarray(b, dtype=np.int64).copy()
        best = np.full(a.shape, -np.inf)
        swap = self.depth[a] < self.depth[b]
        a[swap], b[swap] = b[swap], a[swap].copy()
        diff = self.depth[a] - self.depth[b]
        for j in range(self.L):
            sel = (diff >> j) & 1 == 1
            best[sel] = np.maximum(best[sel], self.mx[j][a[sel]])
            a[sel] = self.up[j][a[sel]]
        for j in range(self.L - 1, -1, -1):
            sel = self.up[j][a] != self.up[j][b]
            best[sel] = np.maximum(best[sel], np.maximum(self.mx[j][a[sel]], self.mx[j][b[sel]]))
            a[sel] = self.up[j][a[sel]]
            b[sel] = self.up[j][b[sel]]
        neq = a != b
        best[neq] = np.maximum(best[neq], np.maximum(self.mx[0][a[neq]], self.mx[0][b[neq]]))
        return best


def check_tree_structure(n, g_lo, g_hi, g_w, where=""):
    g_lo = np.asarray(g_lo, dtype=np.int64)
    g_hi = np.asarray(g_hi, dtype=np.int64)
    g_w = np.asarray(g_w, dtype=np.float64)
    assert g_lo.shape == (max(n - 1, 0),), f"{where}: {g_lo.shape[0]} edges for n = {n}"
    if n <= 1:
        return
    assert (g_lo < g_hi).all() and (g_lo >= 0).all() and (g_hi < n).all(), f"{where}: bad endpoints"
    parent = np.arange(n)

    def find(x):
        while parent[x] != x:
            parent[x] = parent[parent[x]]
            x = parent[x]
        return x

    for a, b in zip(g_lo.tolist(), g_hi.tolist()):
        ra, rb = find(a), find(b)
        assert ra != rb, f"{where}: edge ({a}, {b}) closes a cycle"
        parent[ra] = rb
    keys = np.lexsort((g_hi, g_lo, g_w))
    assert (keys == np.arange(n - 1)).all(), f"{where}: edges not ordered by (w, lo, hi)"


def check_mst(n, g_lo, g_hi, g_w, o_lo, o_hi, o_w, o_weight_of, core_floor, rtol=RTOL, where=""):
    """``o_weight_of(a, b)``: oracle float64 mutual-reachability weight of pairs."""
    check_tree_structure(n, g_lo, g_hi, g_w, where)
    if n <= 1:
        return
    g_lo = np.asarray(g_lo, dtype=np.int64)
    g_hi = np.asarray(g_hi, dtype=np.int64)
    g_w = np.asarray(g_w, dtype=np.float64)
    ow_g = o_weight_of(g_lo, g_hi)
    bad = np.abs(g_w - ow_g) > rtol * ow_g + core_floor
    assert not bad.any(), (f"{where}: edge weights off at {np.flatnonzero(bad)[:5].tolist()}: "
                           f"{g_w[bad][:5]} vs {ow_g[bad][:5]}")
    tg, to = g_w.sum(), float(np.sum(o_w))
    assert abs(tg - to) <= rtol * to, f"{where}: total weight {tg} vs oracle {to}"
    gset = set(zip(g_lo.tolist(), g_hi.tolist()))
    oset = set(zip(np.asarray(o_lo).tolist(), np.asarray(o_hi).tolist()))
    only_g = np.array(sorted(gset - oset), dtype=np.int64).reshape(-1, 2)
    only_o = np.array(sorted(oset - gset), dtype=np.int64).reshape(-1, 2)
    if only_g.size:
        ot = Forest(n, o_lo, o_hi, o_w)
        pm = ot.path_max(only_g[:, 0], only_g[:, 1])
        wg = o_weight_of(only_g[:, 0], only_g[:, 1])
        bad = pm < wg * (1 - rtol)
        assert not bad.any(), (f"{where}: {int(bad.sum())} CUDA edges are not near-tie exchanges, "
                               f"e.g. {only_g[bad][:3].tolist()} w={wg[bad][:3]} path max {pm[bad][:3]}")
    if only_o.size:
        gt = Forest(n, g_lo, g_hi, ow_g)
        pm = gt.path_max(only_o[:, 0], only_o[:, 1])
        wo = o_weight_of(only_o[:, 0], only_o[:, 1])
        bad = pm > wo * (1 + rtol)
        assert not bad.any(), (f"{where}: {int(bad.sum())} oracle edges beat the CUDA tree's path, "
                               f"e.g. {only_o[bad][:3].tolist()}")
    return len(only_g)
