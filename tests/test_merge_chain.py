"""The merge on its worst case: one hook chain through every point.

Page "HDBSCAN", "The algorithm on the device": each round finds every
component's cheapest edge, "then merge"; section "The hang": every loop on the
device is bounded.  The chain set (``chain_points``) makes the first round
hook point i onto point i - 1 for every i, so the hook forest is one path of
depth n - 1.  A root walk costs O(depth) per component there (O(n^2) in all);
the library's pointer jumping needs a number of launches logarithmic in n.
"""

import numpy as np
import pytest

import chain_points
import oracle
from gpu_common import H, dev, np_


def test_chain_tree_is_the_path_oracle():
    """Pin of the construction (no GPU): on a prefix with several turns of
    the path, the oracle's core distances and Prim tree are the closed form,
    the path with weights sqrt(G0 + i)."""
    n = 1500
    X = chain_points.chain(n, row=300)
    P = X.T.astype(np.float64)
    steps = ((P[1:] - P[:-1]) ** 2).sum(axis=1)
    assert np.array_equal(steps, chain_points.G0 + np.arange(1, n))
    oc = oracle.core_distances(X, 2)
    i = np.arange(1, n)
    want_core = np.sqrt((chain_points.G0 + np.concatenate([[1], i])).astype(np.float64))
    assert np.array_equal(oc, want_core)
    lo, hi, w = oracle.prim_mst(X, oc)
    assert np.array_equal(lo, i - 1) and np.array_equal(hi, i)
    assert np.array_equal(w, np.sqrt((chain_points.G0 + i).astype(np.float64)))
    # the float32 closed form the CUDA path must match bit for bit
    clo, chi, cw = chain_points.tree(n)
    assert np.array_equal(clo, lo) and np.array_equal(chi, hi)
    assert np.all(np.abs(cw.astype(np.float64) - w) <= 2.0 ** -24 * w)


def _merge_ms(h, X, ms):
    Xd = dev(X)
    core, idx, dist = h.core_distances(Xd, ms)
    h.profile_read()
    h.profile_enable(True)
    try:
        edges, w = h.mr_mst(Xd, core, idx, dist)
        prof = h.profile_read()
    finally:
        h.profile_enable(False)
    merge = sum(prof.get(k, (0.0, 0))[0] for k in ("hook", "roots", "relabel"))
    return np_(core), np_(edges), np_(w), merge, prof


@pytest.mark.gpu
def test_chain_120k_merge_is_bounded():
    """120 000 points whose first round hooks them into one chain: the tree is
    the path, bit for bit; it takes one round; and the merge (hook, roots,
    relabel) costs no more than twice the merge of a clustered set of the same
    size (plus 0.2 ms of launch noise)."""
    h = H()
    n = 120_000
    X = chain_points.chain(n)
    core, edges, w, merge, prof = _merge_ms(h, X, 2)
    lo, hi, cw = chain_points.tree(n)
    i = np.arange(1, n)
    want_core = np.sqrt((chain_points.G0 + np.concatenate([[1], i])).astype(np.float32))
    assert np.array_equal(core, want_core)
    assert np.array_equal(edges[:, 0], lo) and np.array_equal(edges[:, 1], hi)
    assert np.array_equal(w, cw)
    rounds = h.last_mst_rounds()
    assert len(rounds) == 1 and rounds[0][1] == n - 1, rounds
    import workloads
    Y = workloads.small(n, 6, seed=5, clusters=20)
    _, _, _, merge_ref, _ = _merge_ms(h, Y, 2)
    print(f"merge: chain {merge:.3f} ms, clustered {merge_ref:.3f} ms; {prof}")
    assert merge <= 2.0 * merge_ref + 0.2, (merge, merge_ref)
