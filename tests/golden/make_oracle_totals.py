"""Write ``oracle_totals.json``: the oracle's MST total weight and core-distance
sum for the HDBSCAN workloads, with a digest of the drawn points.

Calls only ``oracle/`` and ``workloads``.  The parity tests compare the CUDA
path's totals with these numbers when the machine draws the same points (same
digest); otherwise they recompute what they need.

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


def main(names):
    data = json.load(open(OUT)) if os.path.exists(OUT) else {}
    for name in names:
        X, task = workloads.workload(name)
        ms = task["min_samples"]
        t0 = time.time()
        core = oracle.core_distances(X, ms)
        t1 = time.time()
        lo, hi, w = oracle.prim_mst(X, core)
        t2 = time.time()
        data[name] = {
            "digest": workloads.digest(X),
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
        print(name, data[name], flush=True)
        json.dump(data, open(OUT, "w"), indent=1, sort_keys=True)


if __name__ == "__main__":
    main(sys.argv[1:] or [k for k, v in workloads.WORKLOADS.items() if v["task"] == "mst"])
