"""Shared pieces of the GPU parity tests."""

import json
import os

import numpy as np
import pytest

import oracle
import parity
import workloads

HERE = os.path.dirname(os.path.abspath(__file__))
TOTALS = os.path.join(HERE, "golden", "oracle_totals.json")


def H():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    from hdbscan_mst_gb300 import build
    build.build()
    import hdbscan_mst_gb300
    return hdbscan_mst_gb300


def dev(X):
    import torch
    return torch.from_numpy(np.ascontiguousarray(X)).cuda()


def np_(t):
    return t.cpu().numpy()


def oracle_knn_check(X, Y, k, g_idx, g_dist, rows=None, where=""):
    """Compare CUDA k-NN rows (all, or the listed ``rows``) with the oracle."""
    m = Y.shape[1]
    Xq = X if rows is None else np.ascontiguousarray(X[:, rows])
    kk = min(k + 1, m)
    oi, od = oracle.knn(Xq, Y, kk)
    gi = np.asarray(g_idx)
    gd = np.asarray(g_dist)
    if rows is not None:
        gi, gd = gi[rows], gd[rows]

    def pd(r, c):
        return oracle.pair_dist_xy(Xq, Y, r, c)

    parity.check_knn(gi, gd, oi, od, k, m, pd, where=where)


def golden_total(name, X):
    """The stored oracle totals of a workload.  A machine that draws other
    points than the ones the oracle ran on fails here: the stored values
    would not apply, and a silent skip would hide the missing check."""
    g = json.load(open(TOTALS))[name]
    assert g["digest"] == workloads.digest(X), (
        f"{name}: this machine drew other points than the stored oracle outputs were made from")
    return g


def golden_outputs(name, X):
    """The oracle's stored whole output of a 200 000-point workload
    (``tests/golden/oracle_<name>.npz``, written by ``make_oracle_totals.py``
    with the oracle alone); fails on a digest mismatch like golden_total."""
    z = np.load(os.path.join(HERE, "golden", f"oracle_{name}.npz"))
    assert str(z["digest"]) == workloads.digest(X), (
        f"{name}: this machine drew other points than the stored oracle outputs were made from")
    return {k: z[k] for k in z.files}
