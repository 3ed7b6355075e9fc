"""Pins of the bipartite assignment oracle (oracle/bipartite.py), no GPU.

Page "Kilosort4 clustering and matching", section "Assignment in parallel:
why the graph is bipartite".  The oracle is checked against values worked
out by hand below, against a plurality vote written with collections.Counter
(gamma = 0 makes the score the neighbour count alone), against the gain
n_vc - gamma k_v K_c / 2m evaluated exactly with fractions, and against the
fixed-point property of its result; and planted mistakes in copies of its
steps must each fail one of these pins.
"""

from collections import Counter
from fractions import Fraction

import numpy as np
import pytest

from oracle import bipartite as B


# ---------------------------------------------------------------- hand-worked

def test_two_blocks():
    """Spikes 0-2 list subset points 0 and 1, spikes 3-5 list 2 and 3; the
    subset starts labelled (0, 0, 1, 1).  Every spike takes its block's
    label (one candidate each), the subset keeps its labels, and the second
    round moves nothing."""
    nbr = np.array([[0, 1]] * 3 + [[2, 3]] * 3)
    left, right, rounds, moved = B.assign(nbr, 4, [0, 0, 1, 1], 2)
    assert left.tolist() == [0, 0, 0, 1, 1, 1]
    assert right.tolist() == [0, 0, 1, 1]
    assert rounds == 2 and moved == [6, 0]


NBR_C = np.array([[0, 1, 2], [0, 1, 3], [0, 1, 3], [0, 1, 3]])


def test_resolution_flips_a_spike():
    """4 spikes, k = 3, subset labels (0, 0, 1, 0); edges 12, 2m = 24;
    right degrees (4, 4, 1, 3); masses K_0 = 11, K_1 = 1.  Spike 0 sees
    label 0 twice and label 1 once: scores 48 - 33 gamma and 24 - 3 gamma, so
    label 1 wins exactly when gamma > 0.8.  The other spikes see label 0 only.

    gamma = 1: spikes (1, 0, 0, 0).  Right step: K_0 = 9, K_1 = 3; point 0
    sees spike labels 1, 0, 0, 0: 72 - 36 = 36 against 24 - 12 = 12, stays 0;
    point 1 likewise; point 2 sees only spike 0 (label 1); point 3 only 0s.
    gamma = 1/2: every spike takes 0; point 2 then sees only label 0."""
    left, right, rounds, moved = B.assign(NBR_C, 4, [0, 0, 1, 0], 2, gamma=1.0)
    assert left.tolist() == [1, 0, 0, 0] and right.tolist() == [0, 0, 1, 0]
    assert rounds == 2 and moved == [4, 0]
    left, right, rounds, moved = B.assign(NBR_C, 4, [0, 0, 1, 0], 2, gamma=0.5)
    assert left.tolist() == [0, 0, 0, 0] and right.tolist() == [0, 0, 0, 0]
    assert rounds == 2


def test_scores_by_hand():
    # spike 0 of the case above: 2m = 24, k = 3, K = (11, 1)
    assert B.scores(24, [2, 1], 3, [11, 1], 1.0).tolist() == [15.0, 21.0]
    assert B.scores(24, [2, 1], 3, [11, 1], 0.5).tolist() == [31.5, 22.5]
    assert B.scores(24, [2, 1], 3, [11, 1], 0.0).tolist() == [48.0, 24.0]


def test_ties():
    """Equal counts: with gamma = 0 the lower label wins; with gamma > 0 the
    lighter cluster wins.  Spike 0 lists subset points 0 (label 3) and 1
    (label 1); spikes 1, 2 list point 1 and 2 (label 1), so K_1 = 3 + 2 = 5 > K_3 = 1."""
    nbr = np.array([[0, 1], [1, 2], [1, 2]])
    deg = B.degrees(nbr, 3)
    assert deg.tolist() == [1, 3, 2]
    right = np.array([3, 1, 1])
    assert B.left_step(nbr, right, deg, 4, 0.0).tolist() == [1, 1, 1]
    # gamma = 1: 2m = 12; label 3: 12 - 2*1 = 10; label 1: 12 - 2*5 = 2
    assert B.left_step(nbr, right, deg, 4, 1.0).tolist() == [3, 1, 1]


def test_only_neighbour_labels_are_candidates():
    """Three spikes list subset points 0 and 1, all labelled 0; cluster 1 is
    empty.  gamma = 3: 2m = 12, K_0 = 6, and point 0's one candidate scores
    36 - 3 * 3 * 6 = -18 < 0, below the 0 an empty cluster would score; it
    stays in cluster 0 all the same."""
    nbr = np.array([[0, 1]] * 3)
    left, right, rounds, _ = B.assign(nbr, 2, [0, 0], 2, gamma=3.0)
    assert left.tolist() == [0, 0, 0] and right.tolist() == [0, 0] and rounds == 2


def test_isolated_subset_point_keeps_its_label():
    nbr = np.array([[0, 1], [0, 1]])
    left, right, rounds, _ = B.assign(nbr, 3, [2, 2, 1], 3)
    assert right[2] == 1 and left.tolist() == [2, 2]


# ---------------------------------------------------------------- other formulations

def random_graph(rng, n, m, k, C):
    nbr = np.stack([rng.choice(m, k, replace=False) for _ in range(n)])
    right = rng.integers(0, C, m)
    return nbr, right


def plurality_left(nbr, right):
    out = []
    for row in nbr:
        c = Counter(int(right[r]) for r in row)
        top = max(c.values())
        out.append(min(l for l, v in c.items() if v == top))
    return out


def plurality_right(nbr, left, right, m):
    lists = [[] for _ in range(m)]
    for t, row in enumerate(nbr):
        for r in row:
            lists[int(r)].append(int(left[t]))
    out = []
    for r in range(m):
        if not lists[r]:
            out.append(int(right[r]))
            continue
        c = Counter(lists[r])
        top = max(c.values())
        out.append(min(l for l, v in c.items() if v == top))
    return out


@pytest.mark.parametrize("seed", range(6))
def test_gamma_zero_is_a_plurality_vote(seed):
    rng = np.random.default_rng(seed)
    nbr, right = random_graph(rng, 50, 30, 5, 6)
    deg = B.degrees(nbr, 30)
    left = B.left_step(nbr, right, deg, 6, 0.0)
    assert left.tolist() == plurality_left(nbr, right)
    assert B.right_step(nbr, left, right, deg, 6, 0.0).tolist() == plurality_right(nbr, left, right, 30)


def exact_best(counts, k_v, K, gamma, two_m):
    """argmax over the candidate labels of n - gamma k_v K_c / 2m, exactly."""
    g = Fraction(gamma)
    best, arg = None, None
    for c in sorted(counts):
        v = Fraction(counts[c]) - g * k_v * K[c] / two_m
        if best is None or v > best:
            best, arg = v, c
    return arg


@pytest.mark.parametrize("gamma", [0.25, 0.5, 1.0, 2.0, 3.0])
@pytest.mark.parametrize("seed", range(4))
def test_steps_against_exact_gain(gamma, seed):
    rng = np.random.default_rng(100 + seed)
    n, m, k, C = 60, 25, 4, 7
    nbr, right = random_graph(rng, n, m, k, C)
    two_m = 2 * n * k
    deg = [0] * m
    for row in nbr:
        for r in row:
            deg[int(r)] += 1
    KR = [0] * C
    for r in range(m):
        KR[int(right[r])] += deg[r]
    want_left = [exact_best(Counter(int(right[r]) for r in row), k, KR, gamma, two_m) for row in nbr]
    left = B.left_step(nbr, right, B.degrees(nbr, m), C, gamma)
    assert left.tolist() == want_left
    KL = [0] * C
    for t in range(n):
        KL[int(left[t])] += k
    want_right = []
    for r in range(m):
        c = Counter(int(left[t]) for t in range(n) if r in nbr[t])
        want_right.append(exact_best(c, deg[r], KL, gamma, two_m) if c else int(right[r]))
    assert B.right_step(nbr, left, right, B.degrees(nbr, m), C, gamma).tolist() == want_right


@pytest.mark.parametrize("gamma", [0.5, 1.0])
@pytest.mark.parametrize("seed", range(4))
def test_result_is_a_fixed_point(gamma, seed):
    rng = np.random.default_rng(200 + seed)
    nbr, right0 = random_graph(rng, 300, 60, 6, 12)
    left, right, rounds, moved = B.assign(nbr, 60, right0, 12, gamma)
    assert moved[-1] == 0 and rounds < 200
    deg = B.degrees(nbr, 60)
    assert np.array_equal(B.left_step(nbr, right, deg, 12, gamma), left)
    assert np.array_equal(B.right_step(nbr, left, right, deg, 12, gamma), right)
    assert deg.sum() == 300 * 6
    assert B.cluster_mass(right, deg, 12).sum() == 300 * 6


# ---------------------------------------------------------------- planted mistakes

def pins_pass():
    try:
        test_two_blocks()
        test_resolution_flips_a_spike()
        test_scores_by_hand()
        test_ties()
        test_only_neighbour_labels_are_candidates()
        test_isolated_subset_point_keeps_its_label()
        for s in range(3):
            test_gamma_zero_is_a_plurality_vote(s)
            for g in (0.5, 1.0, 2.0):
                test_steps_against_exact_gain(g, s)
    except AssertionError:
        return False
    return True


def _same_side_mass_right_step(nbr, left, right, deg_r, C, gamma):
    # mistake: the subset's own masses instead of the spikes'
    nbr = np.asarray(nbr, dtype=np.int64)
    n, k = nbr.shape
    m = deg_r.shape[0]
    K = B.cluster_mass(right, deg_r, C)
    cnt = np.zeros((m, C), dtype=np.int64)
    np.add.at(cnt, (nbr.ravel(), np.repeat(np.asarray(left, dtype=np.int64), k)), 1)
    s = np.where(cnt > 0, B.scores(2 * n * k, cnt, deg_r[:, None], K[None, :], gamma), -np.inf)
    return np.where(deg_r > 0, np.argmax(s, axis=1), right)


def _scores_one_m(two_m, n_vc, k_v, K_c, gamma):
    return _orig_scores(two_m // 2, n_vc, k_v, K_c, gamma)


def _scores_no_gamma(two_m, n_vc, k_v, K_c, gamma):
    return _orig_scores(two_m, n_vc, k_v, K_c, 1.0)


def _left_highest_on_ties(nbr, right, deg_r, C, gamma):
    nbr = np.asarray(nbr, dtype=np.int64)
    n, k = nbr.shape
    K = B.cluster_mass(right, deg_r, C)
    L = np.asarray(right, dtype=np.int64)[nbr]
    cnt = (L[:, :, None] == L[:, None, :]).sum(axis=2)
    s = B.scores(2 * n * k, cnt, k, K[L], gamma)
    return np.where(s == s.max(axis=1, keepdims=True), L, -1).max(axis=1)


def _right_all_clusters(nbr, left, right, deg_r, C, gamma):
    nbr = np.asarray(nbr, dtype=np.int64)
    n, k = nbr.shape
    m = deg_r.shape[0]
    K = B.cluster_mass(left, np.full(n, k, dtype=np.int64), C)
    cnt = np.zeros((m, C), dtype=np.int64)
    np.add.at(cnt, (nbr.ravel(), np.repeat(np.asarray(left, dtype=np.int64), k)), 1)
    s = B.scores(2 * n * k, cnt, deg_r[:, None], K[None, :], gamma)
    return np.where(deg_r > 0, np.argmax(s, axis=1), right)


_orig_scores = B.scores


@pytest.mark.parametrize("name, attr, bad", [
    ("mass from the same side", "right_step", _same_side_mass_right_step),
    ("m instead of 2m", "scores", _scores_one_m),
    ("gamma ignored", "scores", _scores_no_gamma),
    ("highest label on ties", "left_step", _left_highest_on_ties),
    ("every cluster a candidate", "right_step", _right_all_clusters),
])
def test_planted_mistakes_fail_a_pin(monkeypatch, name, attr, bad):
    assert pins_pass()
    monkeypatch.setattr(B, attr, bad)
    assert not pins_pass(), name
