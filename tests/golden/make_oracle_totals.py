"""Write the oracle's stored outputs for the full-size workloads.

* ``oracle_totals.json``: the oracle's MST total weight and core-distance sum
  for the HDBSCAN workloads, with a digest of the drawn points.
* ``oracle_<name>.npz`` for the two 200 000-point workloads, so that the
  parity tests can compare the CUDA path's whole output with the oracle's
  without re-running minutes of float64 brute force on the test machine:

  - ``hdbscan_200k_d61``: every core distance (float64) and the whole tree
    as ``(lo, hi)`` int32 in (w, lo, hi) order.  The weights are not stored:
    they are ``max(core_lo, core_hi, dist(lo, hi))`` and the test recomputes
    them with the oracle's own pair distance, which sums the same float64
    terms in the same order as the Prim step (the script checks that the
    recomputed weights equal Prim's bit for bit before it writes the file).
  - ``knn_200k_d192``: the oracle's k + 1 nearest subset columns of every
    row, ``[n, k + 1]`` (uint16 while the subset has at most 65 536 points) in
    (dist, idx) order; the distances are again
    recomputed by the test with the oracle's pair distance (same terms, same
    order as its k-NN), and checked here likewise.

Calls only ``oracle/`` and ``workloads``; no value comes from the CUDA path.

    python tests/golden/make_oracle_totals.py [workload ...]
"""

import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import workloads  # noqa: E402

OUT = os.path.join(HERE, "oracle_totals.json")
# workloads whose whole oracle output is stored
FULL = ("hdbscan_200k_d61", "knn_200k_d192")


def npz_path(name):
    return os.path.join(HERE, f"oracle_{name}.npz")


def mst_workload(name, data):
    X, task = workloads.workload(name)
    ms = task["min_samples"]
    t0 = time.time()
    core = oracle.core_distances(X, ms)
    t1 = time.time()
    lo, hi, w = oracle.prim_mst(X, core)
    t2 = time.time()
    dg = workloads.digest(X)
    data[name] = {
        "digest": dg,
        "n": int(X.shape[1]),
        "d": int(X.shape[0]),
        "min_samples": ms,
        "mst_total": float(np.sum(w)),
        "mst_edges": int(w.shape[0]),
        "mst_max_weight": float(w.max()) if w.size else 0.0,
        "core_sum": float(np.sum(core)),
        "core_median": float(np.median(core)),
        "oracle_seconds": {"core": round(t1 - t0, 2), "prim": round(t2 - t1, 2)},
        "oracle_threads": oracle.threads(),
    }
    if name in FULL:
        rw = oracle.mr_weights(X, core, lo, hi)
        assert np.array_equal(rw, w), "recomputed weights differ from Prim's"
        np.savez_compressed(npz_path(name), digest=np.array(dg), min_samples=np.array(ms),
                            core=core, lo=lo.astype(np.int32), hi=hi.astype(np.int32))


def knn_workload(name, data):
    X, task = workloads.workload(name)
    Y = workloads.subset_columns(X, task["y_stride"])
    k = task["k"]
    t0 = time.time()
    idx, dist = oracle.knn(X, Y, k + 1)
    t1 = time.time()
    n = X.shape[1]
    rd = oracle.pair_dist_xy(X, Y, np.repeat(np.arange(n), k + 1), idx.ravel()).reshape(n, k + 1)
    assert np.array_equal(rd, dist), "recomputed distances differ from the k-NN's"
    dg = workloads.digest(X)
    data[name] = {
        "digest": dg,
        "n": int(n),
        "m": int(Y.shape[1]),
        "d": int(X.shape[0]),
        "k": k,
        "kth_dist_sum": float(np.sum(dist[:, k - 1])),
        "oracle_seconds": {"knn": round(t1 - t0, 2)},
        "oracle_threads": oracle.threads(),
    }
    if name in FULL:
        itype = np.uint16 if Y.shape[1] <= 65536 else np.int32
        np.savez_compressed(npz_path(name), digest=np.array(dg), k=np.array(k),
                            idx=idx.astype(itype))


def main(names):
    data = json.load(open(OUT)) if os.path.exists(OUT) else {}
    for name in names:
        if workloads.WORKLOADS[name]["task"] == "mst":
            mst_workload(name, data)
        else:
            knn_workload(name, data)
        print(name, data[name], flush=True)
        json.dump(data, open(OUT, "w"), indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or [k for k, v in workloads.WORKLOADS.items() if v["task"] == "mst"])
