"""Oracle of the k-NN graph consumer: bipartite modularity assignment.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this module; the library's product path
never imports it.  It shares no code with the CUDA path.

Source: page "Kilosort4 clustering and matching" (neuro-kitchen dsp-kitchen,
gpu/clustering), section "Assignment in parallel: why the graph is
bipartite".  The graph has one left node per spike and one right node per
point of the subset; the k-NN search links every spike to its k nearest
subset points, so each edge joins a left and a right node.  Labels are
cluster numbers.  With the right labels fixed, each left node's best cluster
depends only on its own neighbours, so all left nodes are assigned at once;
then all right nodes, given the left labels; alternately.  A node takes the
cluster maximising n_vc - gamma k_v K_c / 2m; a counter of moved spikes is
read back each round; at most 200 rounds.

Readings of what the page leaves open (each also listed in the design notes):

* edges are unweighted, one per (spike, listed neighbour); m is their count,
  so 2m = 2 n k is the sum of all degrees; k_v is node v's degree (k for a
  spike, the number of spikes listing it for a subset point);
* n_vc counts v's edges to nodes of the other side labelled c, and K_c is the
  degree sum of the OTHER side's nodes labelled c: the side whose labels are
  fixed during the step.  (This is what keeps a node's best cluster a
  function of its own neighbours and the fixed side alone, the page's reason
  for the bipartite form.)
* the candidates of a node are its neighbours' labels, as the left step's
  "counts its neighbours' labels and takes the best"; a node without
  neighbours keeps its label; equal scores go to the lowest cluster number;
* the score is compared as 2m n_vc - gamma (k_v K_c) in float64, the
  products of integers exact, gamma times the integer rounded once and the
  difference rounded once (no fused multiply-add), so that both
  implementations take the same decision (it orders candidates as
  n_vc - gamma k_v K_c / 2m does, up to that rounding);
* a round is a left step, then, unless no spike moved, a right step; the
  first left step counts every spike as moved; the loop ends after the round
  in which no spike moved, or after max_rounds left steps.
"""

from __future__ import annotations

import numpy as np


def degrees(nbr: np.ndarray, m: int) -> np.ndarray:
    """Degree of every right node: how many (spike, neighbour) edges reach it."""
    return np.bincount(np.asarray(nbr, dtype=np.int64).ravel(), minlength=m).astype(np.int64)


def cluster_mass(labels: np.ndarray, deg: np.ndarray, n_clusters: int) -> np.ndarray:
    """K_c: the degree sum of the nodes labelled c (int64, exact)."""
    K = np.zeros(n_clusters, dtype=np.int64)
    np.add.at(K, np.asarray(labels, dtype=np.int64), np.asarray(deg, dtype=np.int64))
    return K


def scores(two_m: int, n_vc, k_v, K_c, gamma: float) -> np.ndarray:
    """2m n_vc - gamma (k_v K_c) in float64 (see the module text)."""
    a = (np.int64(two_m) * np.asarray(n_vc, dtype=np.int64)).astype(np.float64)
    b = np.float64(gamma) * (np.asarray(k_v, dtype=np.int64) * np.asarray(K_c, dtype=np.int64)).astype(np.float64)
    return a - b


def left_step(nbr: np.ndarray, right: np.ndarray, deg_r: np.ndarray, n_clusters: int,
              gamma: float) -> np.ndarray:
    """Every spike's best cluster given the right labels."""
    nbr = np.asarray(nbr, dtype=np.int64)
    n, k = nbr.shape
    two_m = 2 * n * k
    K = cluster_mass(right, deg_r, n_clusters)
    L = np.asarray(right, dtype=np.int64)[nbr]                    # [n, k] neighbour labels
    cnt = (L[:, :, None] == L[:, None, :]).sum(axis=2)           # n_vc of each listed label
    s = scores(two_m, cnt, k, K[L], gamma)                        # [n, k]
    best = s.max(axis=1, keepdims=True)
    return np.where(s == best, L, np.iinfo(np.int64).max).min(axis=1)


def right_step(nbr: np.ndarray, left: np.ndarray, right: np.ndarray, deg_r: np.ndarray,
               n_clusters: int, gamma: float) -> np.ndarray:
    """Every subset point's best cluster given the spikes' labels."""
    nbr = np.asarray(nbr, dtype=np.int64)
    n, k = nbr.shape
    m = deg_r.shape[0]
    two_m = 2 * n * k
    K = cluster_mass(left, np.full(n, k, dtype=np.int64), n_clusters)
    cnt = np.zeros((m, n_clusters), dtype=np.int64)              # n_rc
    np.add.at(cnt, (nbr.ravel(), np.repeat(np.asarray(left, dtype=np.int64), k)), 1)
    s = scores(two_m, cnt, deg_r[:, None], K[None, :], gamma)     # [m, C]
    s = np.where(cnt > 0, s, -np.inf)                             # candidates: neighbours' labels
    new = np.argmax(s, axis=1)                                    # first maximum: lowest label
    return np.where(deg_r > 0, new, np.asarray(right, dtype=np.int64))


def assign(nbr, m: int, right_init, n_clusters: int, gamma: float = 1.0, max_rounds: int = 200):
    """Alternate left and right steps.  Returns ``(left [n], right [m], rounds,
    moved)`` with ``moved`` the spikes each round's left step moved; the last
    entry is 0 when the labels converged within max_rounds."""
    nbr = np.asarray(nbr, dtype=np.int64)
    n, k = nbr.shape
    right = np.asarray(right_init, dtype=np.int64).copy()
    if n and (nbr.min() < 0 or nbr.max() >= m):
        raise ValueError("neighbour index out of range")
    if m and (right.min() < 0 or right.max() >= n_clusters):
        raise ValueError("label out of range")
    deg_r = degrees(nbr, m)
    left = np.full(n, -1, dtype=np.int64)
    moved = []
    for _ in range(max_rounds):
        new_left = left_step(nbr, right, deg_r, n_clusters, gamma)
        moved.append(int(np.count_nonzero(new_left != left)))
        left = new_left
        if moved[-1] == 0:
            break
        right = right_step(nbr, left, right, deg_r, n_clusters, gamma)
    return left, right, len(moved), moved
