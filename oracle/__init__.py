"""Python handle on the float64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use this module; the library's product path
never imports it.  See ``oracle.c`` for what each function computes and which
passage of the pages it follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared"]

_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)


def compile_c(src: str, out: str) -> str:
    """gcc ``src`` into the shared object ``out`` (OpenMP, no fast-math, no FMA contraction)."""
    tmp = out + f".{os.getpid()}.tmp"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_c(SOURCE, _LIB)
    return _LIB


def _fm(X) -> np.ndarray:
    X = np.ascontiguousarray(X, dtype=np.float32)
    if X.ndim != 2:
        raise ValueError("expected a feature-major [d, n] array")
    return X


def _p(a, t):
    return a.ctypes.data_as(t)


class Oracle:
    """The oracle's entry points, loaded from one shared object."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.oracle_threads.restype = ctypes.c_int
        L.oracle_knn.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, _f32p, ctypes.c_int64,
                                 ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i64p, _f64p]
        L.oracle_core_distances.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, _f32p,
                                            ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                            ctypes.c_int, _f64p]
        L.oracle_prim_mst.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                      _f64p, _i64p, _i64p, _f64p]
        L.oracle_pair_dist.argtypes = [_f32p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                       _i64p, _i64p, ctypes.c_int64, _f64p]
        for f in (L.oracle_knn, L.oracle_core_distances, L.oracle_prim_mst, L.oracle_pair_dist):
            f.restype = ctypes.c_int
        self.L = L
        self.path = path

    def threads(self) -> int:
        return self.L.oracle_threads()

    def knn(self, Xq, Y, k: int) -> tuple[np.ndarray, np.ndarray]:
        """k nearest columns of ``Y [d, m]`` for every column of ``Xq [d, nq]``:
        ``(idx int64 [nq, k], dist float64 [nq, k])`` ordered by (dist, idx)."""
        Xq, Y = _fm(Xq), _fm(Y)
        d, nq = Xq.shape
        m = Y.shape[1]
        if Y.shape[0] != d:
            raise ValueError("feature counts differ")
        idx = np.empty((nq, k), dtype=np.int64)
        dist = np.empty((nq, k), dtype=np.float64)
        rc = self.L.oracle_knn(_p(Xq, _f32p), nq, nq, _p(Y, _f32p), m, m, d, k,
                               _p(idx, _i64p), _p(dist, _f64p))
        if rc:
            raise ValueError(f"oracle_knn rejected its arguments ({rc})")
        return idx, dist

    def core_distances(self, X, min_samples: int, rows=None) -> np.ndarray:
        """float64 core distance of every point (or of the points ``rows``)."""
        X = _fm(X)
        d, n = X.shape
        Xq = X if rows is None else np.ascontiguousarray(X[:, np.asarray(rows)])
        nq = Xq.shape[1]
        out = np.empty(nq, dtype=np.float64)
        rc = self.L.oracle_core_distances(_p(Xq, _f32p), nq, nq, _p(X, _f32p), n, n, d,
                                          min_samples, _p(out, _f64p))
        if rc:
            raise ValueError(f"oracle_core_distances rejected its arguments ({rc})")
        return out

    def prim_mst(self, X, core) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
        """Mutual-reachability MST: ``(lo, hi, w)`` sorted by (w, lo, hi), n-1 edges."""
        X = _fm(X)
        d, n = X.shape
        core = np.ascontiguousarray(core, dtype=np.float64)
        if core.shape != (n,):
            raise ValueError("core must have one entry per point")
        ne = max(n - 1, 0)
        lo = np.empty(ne, dtype=np.int64)
        hi = np.empty(ne, dtype=np.int64)
        w = np.empty(ne, dtype=np.float64)
        rc = self.L.oracle_prim_mst(_p(X, _f32p), n, n, d, _p(core, _f64p), _p(lo, _i64p),
                                    _p(hi, _i64p), _p(w, _f64p))
        if rc:
            raise ValueError(f"oracle_prim_mst rejected its arguments ({rc})")
        return lo, hi, w

    def pair_dist(self, X, a, b) -> np.ndarray:
        """float64 Euclidean distance of each pair (a[e], b[e])."""
        X = _fm(X)
        d, n = X.shape
        a = np.ascontiguousarray(a, dtype=np.int64)
        b = np.ascontiguousarray(b, dtype=np.int64)
        out = np.empty(a.shape[0], dtype=np.float64)
        rc = self.L.oracle_pair_dist(_p(X, _f32p), n, n, d, _p(a, _i64p), _p(b, _i64p),
                                     a.shape[0], _p(out, _f64p))
        if rc:
            raise ValueError(f"oracle_pair_dist rejected its arguments ({rc})")
        return out

    def pair_dist_xy(self, Xq, Y, a, b) -> np.ndarray:
        """float64 distance of each pair (column a[e] of Xq, column b[e] of Y)."""
        Xq, Y = _fm(Xq), _fm(Y)
        Z = np.ascontiguousarray(np.concatenate([Xq, Y], axis=1))
        off = Xq.shape[1]
        return self.pair_dist(Z, np.asarray(a, dtype=np.int64), np.asarray(b, dtype=np.int64) + off)

    def mr_weights(self, X, core, a, b) -> np.ndarray:
        """float64 mutual-reachability weight max(core_a, core_b, |a - b|) of each pair;
        ``core`` is indexed by point."""
        core = np.asarray(core, dtype=np.float64)
        a = np.asarray(a, dtype=np.int64)
        b = np.asarray(b, dtype=np.int64)
        return np.maximum(np.maximum(core[a], core[b]), self.pair_dist(X, a, b))


_lock = threading.Lock()
_default: Oracle | None = None


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def threads() -> int:
    return default().threads()


def knn(Xq, Y, k):
    return default().knn(Xq, Y, k)


def core_distances(X, min_samples, rows=None):
    return default().core_distances(X, min_samples, rows)


def prim_mst(X, core):
    return default().prim_mst(X, core)


def pair_dist(X, a, b):
    return default().pair_dist(X, a, b)


def pair_dist_xy(Xq, Y, a, b):
    return default().pair_dist_xy(Xq, Y, a, b)


def mr_weights(X, core, a, b):
    return default().mr_weights(X, core, a, b)
