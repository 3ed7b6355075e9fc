"""The failure paths of the bounds (page "HDBSCAN", section "The hang": every
loop on the device is bounded, so a fault ends in a reported error instead of
a hang), driven on purpose through the library's test hooks.

* A tensor-core tile whose column stream never delivers its first slab: every
  wait on it gives up after a short limit, the kernel winds down and frees its
  tensor memory, the call returns HDBMST_ERR_TIMEOUT, and the next call on
  the same device computes the right answer.
* Boruvka with its rounds capped below what the tree needs, and with the
  merge's pointer jumping capped below the depth of the hook forest: both
  return HDBMST_ERR_NOCONVERGE instead of a wrong tree or a loop.

No test here faults or hangs the GPU: the waits are bounded and the withheld
slab is simply never requested.
"""

import numpy as np
import pytest

import chain_points
import workloads
from gpu_common import H, dev, np_, oracle_knn_check

pytestmark = pytest.mark.gpu

TIMEOUT, NOCONVERGE = 8, 5


@pytest.mark.parametrize("d", [20, 61, 100])
def test_tensor_tile_timeout_then_recovers(d):
    """d = 20: TF32 tile on 32 features; 61: two-part FP16 tile; 100: the
    wide-row TF32 tile (A low parts in shared memory)."""
    h = H()
    X = workloads.small(2000, d, seed=3)
    Xd = dev(X)
    try:
        h.test_set_tc_hooks(wait_ns=5_000_000, withhold_first_slab=True)
        with pytest.raises(h.HdbmstError) as e:
            h.knn(Xd, Xd, 10)
        assert e.value.status == TIMEOUT
    finally:
        h.test_set_tc_hooks()
    gi, gd = h.knn(Xd, Xd, 10)
    oracle_knn_check(X, X, 10, np_(gi), np_(gd), where=f"after timeout, d={d}")


def test_mst_round_cap_reports_noconverge():
    h = H()
    X = workloads.small(3000, 16, seed=4, clusters=6, outlier_frac=0.05)
    Xd = dev(X)
    core, idx, dist = h.core_distances(Xd, 5)
    try:
        h.test_set_mst_caps(max_rounds=1)
        with pytest.raises(h.HdbmstError) as e:
            h.mr_mst(Xd, core, idx, dist)
        assert e.value.status == NOCONVERGE
    finally:
        h.test_set_mst_caps()
    edges, w = h.mr_mst(Xd, core, idx, dist)
    assert edges.shape == (2999, 2) and len(h.last_mst_rounds()) >= 2


def test_merge_jump_cap_reports_noconverge():
    """The chain set hooks 5 000 points into one chain of depth 4 999: one
    launch of 16-step jumps cannot reach the roots, and the merge says so."""
    h = H()
    n = 5000
    X = chain_points.chain(n, row=1000)
    Xd = dev(X)
    core, idx, dist = h.core_distances(Xd, 2)
    try:
        h.test_set_mst_caps(max_jump_launches=1)
        with pytest.raises(h.HdbmstError) as e:
            h.mr_mst(Xd, core, idx, dist)
        assert e.value.status == NOCONVERGE
    finally:
        h.test_set_mst_caps()
    edges, w = h.mr_mst(Xd, core, idx, dist)
    lo, hi, cw = chain_points.tree(n)
    e = np_(edges)
    assert np.array_equal(e[:, 0], lo) and np.array_equal(e[:, 1], hi)
    assert np.array_equal(np_(w), cw)
