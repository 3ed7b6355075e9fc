"""Oracle for the HDBSCAN back half: the cluster hierarchy of the minimum
spanning tree, its condensed tree, excess-of-mass selection and labels.

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU-baseline leg use
this module; the library's product path never imports it.  Plain Python over
lists and dicts, written for reading, not speed.

Source: page "HDBSCAN" (neuro-kitchen dsp-kitchen gpu/hdbscan), "The
algorithm on the device": after the spanning tree, the hierarchy, its
condensed tree and the excess-of-mass selection run on the host; the
introduction says the upstream sorter runs scikit-learn's HDBSCAN.  The page
gives no further detail, so this module states the standard definitions that
scikit-learn's HDBSCAN implements (the plainest reading), with these
choices made explicit:

* min_cluster_size only (no cluster-size cap, no selection epsilon), the root
  is never selected (no single-cluster result);
* the single-linkage merge for edge (lo, hi, w) takes the component of lo as
  its first child and that of hi as its second; the condensed tree is built
  breadth-first, first child before second; stabilities are accumulated in
  the order the condensed tree's entries are made (the order fixes the float
  rounding of the sums, so the library does the same);
* lambda = 1 / w, infinite for w = 0;
* labels: clusters are numbered 0, 1, ... in ascending order of their
  smallest point index; noise is -1.
"""

from __future__ import annotations

import math
from collections import deque

import numpy as np


def single_linkage(n, lo, hi, w):
    """Merge tree of the edges taken in the given (ascending weight) order.

    Returns (first, second, dist, size) lists for the internal nodes n .. 2n-2:
    node n + i merges the components of lo[i] and hi[i] at distance w[i]."""
    parent = list(range(2 * n - 1 if n > 0 else 0))

    def find(x):
        root = x
        while parent[root] != root:
            root = parent[root]
        while parent[x] != root:
            parent[x], x = root, parent[x]
        return root

    size = [1] * n + [0] * max(n - 1, 0)
    first, second, dist = [], [], []
    for i in range(n - 1):
        a, b = find(int(lo[i])), find(int(hi[i]))
        if a == b:
            raise ValueError("the edges do not form a spanning tree")
        node = n + i
        parent[a] = node
        parent[b] = node
        size[node] = size[a] + size[b]
        first.append(a)
        second.append(b)
        dist.append(float(w[i]))
    return first, second, dist, size


def _lam(d):
    return 1.0 / d if d > 0.0 else math.inf


def condense(n, tree, min_cluster_size):
    """Condensed tree entries (parent cluster, child, lambda, child size).

    Clusters are labelled n (the root), n + 1, ... in the order they appear;
    children below n are points."""
    first, second, dist, size = tree
    if n < 2:
        return []
    root = 2 * n - 2

    def children(node):
        return first[node - n], second[node - n]

    def leaves(node):
        out, queue = [], deque([node])
        while queue:
            x = queue.popleft()
            if x < n:
                out.append(x)
            else:
                queue.extend(children(x))
        return out

    relabel = {root: n}
    next_label = n + 1
    entries = []
    queue = deque([root])
    while queue:
        node = queue.popleft()
        if node < n:
            continue
        a, b = children(node)
        lam = _lam(dist[node - n])
        sa, sb = size[a], size[b]
        me = relabel[node]
        if sa >= min_cluster_size and sb >= min_cluster_size:
            for c, sc in ((a, sa), (b, sb)):
                relabel[c] = next_label
                next_label += 1
                entries.append((me, relabel[c], lam, sc))
                queue.append(c)
        elif sa < min_cluster_size and sb < min_cluster_size:
            for c in (a, b):
                for p in leaves(c):
                    entries.append((me, p, lam, 1))
        elif sa < min_cluster_size:
            for p in leaves(a):
                entries.append((me, p, lam, 1))
            relabel[b] = me
            queue.append(b)
        else:
            for p in leaves(b):
                entries.append((me, p, lam, 1))
            relabel[a] = me
            queue.append(a)
    return entries


def stabilities(n, entries):
    """Stability of every cluster: the sum over its entries of
    (lambda - its birth lambda) x child size, the root born at 0."""
    birth = {n: 0.0}
    for parent, child, lam, _ in entries:
        if child >= n:
            birth[child] = lam
    stab = {c: 0.0 for c in birth}
    for parent, child, lam, sz in entries:
        stab[parent] += (lam - birth[parent]) * sz
    return stab


def select_eom(n, entries, stab):
    """Excess of mass: bottom-up, a cluster is kept when its stability is at
    least the summed (already resolved) stability of its child clusters, and
    then replaces every kept cluster below it.  The root is not a candidate."""
    kids = {}
    for parent, child, _, _ in entries:
        if child >= n:
            kids.setdefault(parent, []).append(child)
    stab = dict(stab)
    chosen = set()
    for node in sorted(stab, reverse=True):
        if node == n:
            continue
        below = sum(stab[c] for c in kids.get(node, []))
        if below > stab[node]:
            stab[node] = below
        else:
            chosen.add(node)
            stack = list(kids.get(node, []))
            while stack:
                c = stack.pop()
                chosen.discard(c)
                stack.extend(kids.get(c, []))
    return chosen


def labels_of(n, entries, chosen):
    """Each point's nearest chosen ancestor in the condensed tree, numbered
    by ascending smallest point index; -1 where there is none."""
    up = {}
    for parent, child, _, _ in entries:
        up[child] = parent
    raw = []
    for p in range(n):
        c = up.get(p)
        while c is not None and c not in chosen:
            c = up.get(c)
        raw.append(c)
    first_point = {}
    for p, c in enumerate(raw):
        if c is not None and c not in first_point:
            first_point[c] = p
    order = sorted(first_point, key=lambda c: first_point[c])
    number = {c: i for i, c in enumerate(order)}
    return np.array([number[c] if c is not None else -1 for c in raw], dtype=np.int64)


def hdbscan_labels(n, lo, hi, w, min_cluster_size):
    """Labels of the n points from their minimum spanning tree, edges in
    (w, lo, hi) order."""
    if n == 1:
        return np.array([-1], dtype=np.int64)
    if n == 0:
        return np.zeros(0, dtype=np.int64)
    tree = single_linkage(n, lo, hi, w)
    entries = condense(n, tree, min_cluster_size)
    stab = stabilities(n, entries)
    chosen = select_eom(n, entries, stab)
    return labels_of(n, entries, chosen)
