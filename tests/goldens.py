"""Reader for the hand-worked fixtures in ``tests/golden/*.txt``.

Each fixture is ``key: values`` lines with ``#`` comments (the comments carry
the citation).  Numbers may be written as plain decimals, ``sqrt(x)``, or sums
and products of those (``5 + sqrt(2) + 2*sqrt(10)``).
"""

from __future__ import annotations

import glob
import math
import os
import re

import numpy as np

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

_NUM = re.compile(r"^[0-9.\s+*()sqrt\-]+$")


def _value(tok: str) -> float:
    tok = tok.strip()
    if not _NUM.match(tok):
        raise ValueError(f"not a number expression: {tok!r}")
    return float(eval(tok, {"__builtins__": {}}, {"sqrt": math.sqrt}))


def _values(s: str) -> list[float]:
    # split on whitespace that is not inside parentheses
    out, depth, cur = [], 0, ""
    for ch in s.strip():
        if ch == "(":
            depth += 1
        elif ch == ")":
            depth -= 1
        if ch.isspace() and depth == 0:
            if cur:
                out.append(cur)
            cur = ""
        else:
            cur += ch
    if cur:
        out.append(cur)
    return [_value(t) for t in out]


def load(path: str) -> dict:
    g: dict = {"points": [], "knn": [], "knn_dist": [], "edges": []}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(":")
        key = key.strip()
        if key == "name":
            g["name"] = rest.strip()
        elif key in ("dim", "min_samples", "knn_k", "min_cluster_size"):
            g[key] = int(rest)
        elif key == "labels":
            g["labels"] = np.array([int(v) for v in rest.split()], dtype=np.int64)
        elif key == "point":
            g["points"].append(_values(rest))
        elif key == "core":
            g["core"] = np.array(_values(rest))
        elif key == "knn":
            g["knn"].append([int(v) for v in _values(rest)])
        elif key == "knn_dist":
            g["knn_dist"].append(_values(rest))
        elif key == "edge":
            a, b, w = _values(rest)
            g["edges"].append((int(a), int(b), w))
        elif key == "total":
            g["total"] = _value(rest)
        else:
            raise ValueError(f"{path}: unknown key {key!r}")
    X = np.array(g["points"], dtype=np.float32).T  # [d, n]
    assert X.shape[0] == g["dim"], path
    g["X"] = np.ascontiguousarray(X)
    return g


def all_fixtures() -> list[dict]:
    return [load(p) for p in sorted(glob.glob(os.path.join(GOLDEN_DIR, "*.txt")))]
