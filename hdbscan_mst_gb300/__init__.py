"""GB300-native exact k-NN, HDBSCAN core distances and mutual-reachability MST.

A thin Python binding over the C ABI of ``libhdbmst.so`` (declared in
``include/hdbmst.h``): it checks shapes, allocates outputs and the workspace
with PyTorch on the device, and passes raw pointers and the current CUDA
stream.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU path.  If the library has not been built or cannot be loaded
the functions raise ``HdbmstUnavailable``.

Point sets are float32, feature-major ``[d, n]`` (each row one feature, each
column one point), as torch CUDA tensors with unit column stride.  Host inputs
(numpy arrays or CPU tensors) are accepted too: they are copied to the device,
and the results are copied back to the host.
"""

from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

from . import build as _build

__all__ = [
    "knn", "core_distances", "mr_mst", "hdbscan_mst", "HdbmstError", "HdbmstUnavailable",
    "launch_count", "profile_enable", "profile_read", "last_mst_rounds", "library_path", "KMAX",
    "set_engine", "set_scan_form", "set_scan_pruning",
]

KMAX = 32
OP_KNN, OP_CORE, OP_MST, OP_ASSIGN, OP_MOMENT = 0, 1, 2, 3, 4

STATUS = {
    0: "ok", 1: "invalid argument", 2: "unsupported size", 3: "workspace missing or too small",
    4: "non-finite value", 5: "Boruvka made no progress", 6: "CUDA error",
    7: "too large for the fixed scratch", 8: "a wait inside a kernel gave up",
}


class HdbmstError(RuntimeError):
    def __init__(self, status: int, what: str, detail: str = ""):
        self.status = status
        msg = f"{what}: {STATUS.get(status, status)} ({status})"
        super().__init__(msg + (f" [{detail}]" if detail else ""))


class HdbmstUnavailable(ImportError):
    pass


_lib = None


def library_path() -> str:
    return _build.LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        raise HdbmstUnavailable(
            f"{_build.LIB} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"`")
    try:
        L = ctypes.CDLL(_build.LIB)
    except OSError as e:  # pragma: no cover - depends on the machine
        raise HdbmstUnavailable(f"cannot load {_build.LIB}: {e}") from e
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    L.hdbmst_workspace_bytes.argtypes = [i32, i64, i64, i32, i32]
    L.hdbmst_workspace_bytes.restype = sz
    L.hdbmst_knn.argtypes = [vp, i64, i64, vp, i64, i64, i32, i32, vp, vp, vp, sz, vp]
    L.hdbmst_knn.restype = i32
    L.hdbmst_core_distances.argtypes = [vp, i64, i64, i32, i32, vp, vp, vp, vp, sz, vp]
    L.hdbmst_core_distances.restype = i32
    L.hdbmst_mr_mst.argtypes = [vp, i64, i64, i32, vp, vp, vp, i32, vp, vp, vp, sz, vp]
    L.hdbmst_mr_mst.restype = i32
    L.hdbmst_status_string.argtypes = [i32]
    L.hdbmst_status_string.restype = ctypes.c_char_p
    L.hdbmst_version.restype = i32
    L.hdbmst_launch_count.restype = ctypes.c_uint64
    L.hdbmst_profile_enable.argtypes = [i32]
    L.hdbmst_profile_read.argtypes = [ctypes.POINTER(ctypes.c_double),
                                      ctypes.POINTER(ctypes.c_int64), i32]
    L.hdbmst_profile_read.restype = i32
    L.hdbmst_profile_kernel_name.argtypes = [i32]
    L.hdbmst_profile_kernel_name.restype = ctypes.c_char_p
    L.hdbmst_last_mst_rounds.argtypes = [ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_int64),
                                         ctypes.POINTER(ctypes.c_int64), i32]
    L.hdbmst_last_mst_rounds.restype = i32
    L.hdbmst_set_engine.argtypes = [i32]
    L.hdbmst_set_engine.restype = i32
    L.hdbmst_set_scan_list_cap.argtypes = [i64]
    L.hdbmst_set_scan_list_cap.restype = i64
    L.hdbmst_set_scan_pruning.argtypes = [i32]
    L.hdbmst_set_scan_pruning.restype = i32
    L.hdbmst_set_scan_form.argtypes = [i32]
    L.hdbmst_set_scan_form.restype = i32
    L.hdbmst_last_mst_symmetric.argtypes = [ctypes.POINTER(ctypes.c_int64), i32]
    L.hdbmst_last_mst_symmetric.restype = i32
    L.hdbmst_last_cuda_error.restype = ctypes.c_char_p
    L.hdbmst_last_knn_exact_rows.restype = ctypes.c_int64
    L.hdbmst_last_knn_tile_pairs.restype = ctypes.c_int64
    L.hdbmst_last_mst_scan_pairs.restype = ctypes.c_int64
    L.hdbmst_hdbscan_labels.argtypes = [vp, vp, i64, i32, vp]
    L.hdbmst_hdbscan_labels.restype = i32
    L.hdbmst_bipartite_assign.argtypes = [vp, i64, i32, i64, i32, ctypes.c_double, vp, vp, vp,
                                          i32, ctypes.POINTER(i32), vp, sz, vp]
    L.hdbmst_bipartite_assign.restype = i32
    L.hdbmst_last_assign_moved.argtypes = [ctypes.POINTER(ctypes.c_int64), i32]
    L.hdbmst_last_assign_moved.restype = i32
    L.hdbmst_second_moment.argtypes = [vp, i64, i32, i64, i64, i32, i32, vp, vp, sz, vp]
    L.hdbmst_second_moment.restype = i32
    L.hdbmst_test_set_tc_hooks.argtypes = [ctypes.c_uint64, i32]
    L.hdbmst_test_set_tc_hooks.restype = i32
    L.hdbmst_test_set_mst_caps.argtypes = [i32, i32]
    L.hdbmst_test_tmem_max.argtypes = [ctypes.c_void_p]
    L.hdbmst_test_tmem_max.restype = i32
    L.hdbmst_test_set_mst_caps.restype = None
    _lib = L
    return L


def lib():
    """The loaded ctypes library (loads it on first use)."""
    return _load()


def _check(status: int, what: str):
    if status != 0:
        detail = _lib.hdbmst_last_cuda_error().decode() if status == 6 and _lib else ""
        raise HdbmstError(status, what, detail)


# ---------------------------------------------------------------- marshalling

def _device_points(X, name: str):
    """Return (tensor on CUDA [d, n] float32 with unit column stride, was_host)."""
    host = False
    if isinstance(X, np.ndarray):
        X = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32))
        host = True
    if not isinstance(X, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor or numpy array")
    if X.dim() != 2:
        raise ValueError(f"{name} must be feature-major [d, n]")
    if X.device.type != "cuda":
        host = True
        X = X.to(dtype=torch.float32).pin_memory().to("cuda", non_blocking=True)
    if X.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    if X.stride(1) != 1 or (X.shape[0] > 1 and X.stride(0) < X.shape[1]):
        X = X.contiguous()
    return X, host


def _ld(X) -> int:
    return X.stride(0) if X.shape[0] > 1 else max(X.shape[1], 1)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _workspace(nbytes: int, device, workspace=None):
    if nbytes == 0:
        raise HdbmstError(1, "workspace size")
    if workspace is not None:
        if workspace.numel() * workspace.element_size() < nbytes or workspace.data_ptr() % 256:
            raise HdbmstError(3, "caller workspace")
        return workspace
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def _out(t, host):
    return t.cpu() if host else t


# ---------------------------------------------------------------- operations

def knn(X, Y, k: int, *, workspace=None):
    """Exact k nearest columns of ``Y [d, m]`` for every column of ``X [d, n]``.

    Returns ``(idx int32 [n, k], dist float32 [n, k])`` ordered by
    (distance, index); a query that is also in Y finds itself at distance 0.
    """
    L = _load()
    X, hx = _device_points(X, "X")
    Y, hy = _device_points(Y, "Y")
    d, n = X.shape
    if Y.shape[0] != d:
        raise ValueError("X and Y must have the same number of features")
    m = Y.shape[1]
    dev = X.device
    idx = torch.empty((n, k), dtype=torch.int32, device=dev)
    dist = torch.empty((n, k), dtype=torch.float32, device=dev)
    nb = L.hdbmst_workspace_bytes(OP_KNN, n, m, d, k)
    if nb == 0:
        _check(2 if k > KMAX else 1, "knn")
    ws = _workspace(nb, dev, workspace)
    st = L.hdbmst_knn(X.data_ptr(), _ld(X), n, Y.data_ptr(), _ld(Y), m, d, k, idx.data_ptr(),
                      dist.data_ptr(), ws.data_ptr(), nb, _stream())
    _check(st, "hdbmst_knn")
    host = hx or hy
    return _out(idx, host), _out(dist, host)


def core_distances(X, min_samples: int, *, lists: bool = True, workspace=None):
    """HDBSCAN core distances: each point's distance to its min_samples-th
    nearest point, itself counted first.

    Returns ``core float32 [n]`` and, with ``lists=True``, the neighbour lists
    ``(idx int32 [n, L], dist float32 [n, L])`` with ``L = min(min_samples + 1, n)``,
    which :func:`mr_mst` uses for its exact shortcuts.
    """
    L_ = _load()
    X, host = _device_points(X, "X")
    d, n = X.shape
    dev = X.device
    L = min(min_samples + 1, n)
    core = torch.empty(n, dtype=torch.float32, device=dev)
    idx = torch.empty((n, L), dtype=torch.int32, device=dev) if lists else None
    dist = torch.empty((n, L), dtype=torch.float32, device=dev) if lists else None
    nb = L_.hdbmst_workspace_bytes(OP_CORE, n, 0, d, min_samples)
    if nb == 0:
        _check(2 if min_samples + 1 > KMAX and min_samples <= n else 1, "core_distances")
    ws = _workspace(nb, dev, workspace)
    st = L_.hdbmst_core_distances(X.data_ptr(), _ld(X), n, d, min_samples, core.data_ptr(),
                                  idx.data_ptr() if lists else None,
                                  dist.data_ptr() if lists else None, ws.data_ptr(), nb,
                                  _stream())
    _check(st, "hdbmst_core_distances")
    if not lists:
        return _out(core, host)
    return _out(core, host), _out(idx, host), _out(dist, host)


def mr_mst(X, core, knn_idx=None, knn_dist=None, *, workspace=None):
    """Minimum spanning tree of max(core_a, core_b, |a - b|) by Boruvka.

    ``knn_idx``/``knn_dist`` (both or neither): the lists from
    :func:`core_distances` on the same X; they enable the exact shortcuts and
    do not change the result.  Returns ``(edges int32 [n-1, 2], w float32 [n-1])``
    with ``edges[:, 0] < edges[:, 1]``, ordered by (w, lo, hi).
    """
    Lb = _load()
    X, host = _device_points(X, "X")
    d, n = X.shape
    dev = X.device
    core = torch.as_tensor(core, dtype=torch.float32).to(dev).contiguous()
    if core.shape != (n,):
        raise ValueError("core must have one entry per point")
    if (knn_idx is None) != (knn_dist is None):
        raise ValueError("pass both neighbour lists or neither")
    kl = 0
    if knn_idx is not None:
        knn_idx = torch.as_tensor(knn_idx, dtype=torch.int32).to(dev).contiguous()
        knn_dist = torch.as_tensor(knn_dist, dtype=torch.float32).to(dev).contiguous()
        if knn_idx.dim() != 2 or knn_idx.shape[0] != n or knn_dist.shape != knn_idx.shape:
            raise ValueError("neighbour lists must be [n, L]")
        kl = knn_idx.shape[1]
    ne = max(n - 1, 0)
    edges = torch.empty((ne, 2), dtype=torch.int32, device=dev)
    w = torch.empty(ne, dtype=torch.float32, device=dev)
    nb = Lb.hdbmst_workspace_bytes(OP_MST, n, 0, d, kl)
    if nb == 0:
        _check(1, "mr_mst")
    ws = _workspace(nb, dev, workspace)
    st = Lb.hdbmst_mr_mst(X.data_ptr(), _ld(X), n, d, core.data_ptr(),
                          knn_idx.data_ptr() if kl else None, knn_dist.data_ptr() if kl else None,
                          kl, edges.data_ptr(), w.data_ptr(), ws.data_ptr(), nb, _stream())
    _check(st, "hdbmst_mr_mst")
    return _out(edges, host), _out(w, host)


def hdbscan_mst(X, min_samples: int, *, shortcuts: bool = True):
    """Core distances and the mutual-reachability MST of X in one call.

    Returns ``(core [n], edges [n-1, 2], w [n-1])``; host inputs give host outputs.
    """
    X, host = _device_points(X, "X")
    core, idx, dist = core_distances(X, min_samples, lists=True)
    if shortcuts:
        edges, w = mr_mst(X, core, idx, dist)
    else:
        edges, w = mr_mst(X, core)
    return _out(core, host), _out(edges, host), _out(w, host)


def _device_int32(a, name: str):
    """Return (contiguous int32 CUDA tensor, was_host)."""
    host = False
    if isinstance(a, np.ndarray):
        a = torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))
        host = True
    if not isinstance(a, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor or numpy array")
    if a.device.type != "cuda":
        host = True
        a = a.to(dtype=torch.int32).pin_memory().to("cuda", non_blocking=True)
    if a.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return a.contiguous(), host


def bipartite_assign(nbr, m: int, right_init, n_clusters: int, gamma: float = 1.0,
                     max_rounds: int = 200, *, workspace=None):
    """Bipartite modularity assignment over the k-NN graph ``nbr [n, k]``
    (indices into m subset points, as ``knn`` returns them against the
    subset), from the subset's initial labels ``right_init [m]``.

    Returns ``(left int32 [n], right int32 [m], rounds, moved)``: the spikes'
    and the subset's labels, the left steps taken and the spikes each moved
    (the last 0 when the labels converged)."""
    L = _load()
    nb_t, h1 = _device_int32(nbr, "nbr")
    r0, h2 = _device_int32(right_init, "right_init")
    if nb_t.dim() != 2:
        raise ValueError("nbr must be [n, k]")
    n, k = nb_t.shape
    if r0.shape != (m,):
        raise ValueError("right_init must have one label per subset point")
    dev = r0.device
    left = torch.empty(n, dtype=torch.int32, device=dev)
    right = torch.empty(m, dtype=torch.int32, device=dev)
    nb = L.hdbmst_workspace_bytes(OP_ASSIGN, n, m, n_clusters, k)
    if nb == 0:
        _check(2 if (k > KMAX or n_clusters > 65536 or n > (1 << 23)) else 1, "bipartite_assign")
    ws = _workspace(nb, dev, workspace)
    rounds = ctypes.c_int(0)
    st = L.hdbmst_bipartite_assign(nb_t.data_ptr(), n, k, m, n_clusters, float(gamma),
                                   r0.data_ptr(), left.data_ptr(), right.data_ptr(),
                                   int(max_rounds), ctypes.byref(rounds), ws.data_ptr(), nb,
                                   _stream())
    _check(st, "hdbmst_bipartite_assign")
    moved = (ctypes.c_int64 * 1024)()
    r = L.hdbmst_last_assign_moved(moved, 1024)
    host = h1 or h2
    return _out(left, host), _out(right, host), int(rounds.value), [int(moved[i]) for i in range(r)]


def second_moment(X, t0: int = 0, n: int | None = None, *, centred: bool = True, out=None,
                  accumulate: bool = False, workspace=None):
    """Covariance ``(V - mu)(V - mu)^T / n`` (``centred``) or second moment
    ``V V^T / n`` of the window ``V = X[:, t0:t0 + n]`` of a channel-major
    recording ``X [channels, samples]`` (float32).  Returns ``out``
    ``[channels, channels]`` float32 (a new tensor, or the given one, written
    or, with ``accumulate``, added to)."""
    L = _load()
    host = False
    if isinstance(X, np.ndarray):
        X = torch.from_numpy(np.ascontiguousarray(X, dtype=np.float32))
        host = True
    if X.dim() != 2:
        raise ValueError("X must be channel-major [channels, samples]")
    if X.device.type != "cuda":
        host = True
        X = X.to(dtype=torch.float32).contiguous().pin_memory().to("cuda", non_blocking=True)
    if X.dtype != torch.float32:
        raise TypeError("X must be float32")
    if X.stride(1) != 1:
        X = X.contiguous()
    C, T = X.shape
    n = T - t0 if n is None else n
    ld = X.stride(0) if C > 1 else T
    dev = X.device
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an out tensor")
        out = torch.empty((C, C), dtype=torch.float32, device=dev)
    elif out.device.type != "cuda" or out.dtype != torch.float32 or out.shape != (C, C) \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 [channels, channels] CUDA tensor")
    nb = L.hdbmst_workspace_bytes(OP_MOMENT, n, 0, C, 0)
    if nb == 0:
        _check(1, "second_moment")
    ws = _workspace(nb, dev, workspace)
    st = L.hdbmst_second_moment(X.data_ptr(), ld, C, t0, n, 1 if centred else 0,
                                1 if accumulate else 0, out.data_ptr(), ws.data_ptr(), nb,
                                _stream())
    _check(st, "hdbmst_second_moment")
    return _out(out, host)


def hdbscan_labels(edges, w, min_cluster_size: int):
    """HDBSCAN labels from a spanning tree (``hdbmst_hdbscan_labels``, host).

    ``edges [n-1, 2]`` int32 and ``w [n-1]`` float32 as ``mr_mst`` returns them
    (device tensors are copied to the host); returns host ``labels [n]`` int32
    (clusters 0, 1, ... by smallest point index, -1 for noise)."""
    import numpy as np
    E = np.ascontiguousarray(_host_array(edges), dtype=np.int32).reshape(-1, 2)
    W = np.ascontiguousarray(_host_array(w), dtype=np.float32).reshape(-1)
    if E.shape[0] != W.shape[0]:
        raise ValueError("edges and w disagree in length")
    n = E.shape[0] + 1
    labels = np.empty(n, dtype=np.int32)
    st = _load().hdbmst_hdbscan_labels(E.ctypes.data, W.ctypes.data, n, int(min_cluster_size),
                                       labels.ctypes.data)
    _check(st, "hdbmst_hdbscan_labels")
    return labels


def hdbscan(X, min_samples: int, min_cluster_size: int):
    """The whole method: core distances and the MR-MST on the GPU, labels on
    the host.  Returns host ``(labels [n], core [n], edges [n-1, 2], w [n-1])``."""
    core, edges, w = hdbscan_mst(X, min_samples)
    core, edges, w = (_host_array(t) for t in (core, edges, w))
    if edges.shape[0] == 0:
        import numpy as np
        return np.full(core.shape[0], -1, dtype=np.int32), core, edges, w
    return hdbscan_labels(edges, w, min_cluster_size), core, edges, w


def _host_array(t):
    """A numpy view or copy of a numpy array or a (CPU or CUDA) tensor."""
    import numpy as np
    if isinstance(t, np.ndarray):
        return t
    return t.detach().cpu().numpy()


# ---------------------------------------------------------------- instrumentation

ENGINES = {"auto": 0, "simt": 1, "tensor": 2, "tf32": 3}


def set_engine(engine: str) -> str:
    """Select the distance-tile engine ("auto", "simt", "tensor" or "tf32", the
    tensor cores with TF32 products only); returns the previous one.  Results
    are identical whichever engine runs."""
    prev = _load().hdbmst_set_engine(ENGINES[engine])
    return {v: k for k, v in ENGINES.items()}[prev]


SCAN_FORMS = {"auto": 0, "one_sided": 1, "symmetric": 2}


def set_scan_form(form: str) -> str:
    """Select the form of the Boruvka scan on the tensor cores ("auto",
    "one_sided" or "symmetric"); returns the previous one.  The tree is the
    same whichever form runs."""
    prev = _load().hdbmst_set_scan_form(SCAN_FORMS[form])
    return {v: k for k, v in SCAN_FORMS.items()}[prev]


def set_scan_pruning(on: bool) -> bool:
    """Turn the block pruning of the symmetric scan on or off; returns the
    previous setting.  The tree is the same either way."""
    return bool(_load().hdbmst_set_scan_pruning(1 if on else 0))


def set_scan_list_cap(cap: int) -> int:
    """Cap the recorded-pair lists of the symmetric scan and of the open-row
    rescan (0: the default); an overflow sends the round (rows) to the
    one-sided (exact) scan, with the same tree.  Returns the previous cap."""
    return int(_load().hdbmst_set_scan_list_cap(int(cap)))


def test_set_tc_hooks(wait_ns: int = 0, withhold_first_slab: bool = False) -> None:
    """Failure-path test hook, current device: the tensor-core tiles' wait
    limit (0: the default 1.5 s) and whether every tile leaves its first
    column slab unloaded (its waits then run out: HDBMST_ERR_TIMEOUT).
    ``test_set_tc_hooks()`` restores the defaults."""
    _check(_load().hdbmst_test_set_tc_hooks(int(wait_ns), 1 if withhold_first_slab else 0),
           "hdbmst_test_set_tc_hooks")


def test_tmem_max():
    """Hardware check the tensor-core tiles' batch floor rests on (current
    device): a [128, 68] float32 tensor - per TMEM lane its 64 stored values
    read back, then the maxima of columns 0..31 and 32..63 from the
    one-batch and from the two-batch max-reducing loads (the stored values
    are defined in include/hdbmst.h, hdbmst_test_tmem_max)."""
    import torch
    out = torch.empty((128, 68), dtype=torch.float32, device="cuda")
    _check(_load().hdbmst_test_tmem_max(ctypes.c_void_p(out.data_ptr())), "hdbmst_test_tmem_max")
    return out


def test_set_mst_caps(max_rounds: int = 0, max_jump_launches: int = 0) -> None:
    """Failure-path test hook: cap mr_mst's Boruvka rounds and its merge's
    pointer-jumping launches per round (0: no cap, the default)."""
    _load().hdbmst_test_set_mst_caps(int(max_rounds), int(max_jump_launches))


def last_mst_symmetric() -> list[int]:
    """Per Boruvka round of the last mr_mst call: pairs the symmetric scan
    recorded, or -1 for a one-sided round."""
    L = _load()
    a = (ctypes.c_int64 * 64)()
    r = L.hdbmst_last_mst_symmetric(a, 64)
    return [int(a[i]) for i in range(min(r, 64))]


def launch_count() -> int:
    """Kernels the library has launched in this process."""
    return int(_load().hdbmst_launch_count())


def profile_enable(on: bool = True) -> None:
    """Record CUDA events around every kernel launch (on the launching stream)."""
    _load().hdbmst_profile_enable(1 if on else 0)


def last_mst_rounds() -> list[tuple[int, int, int]]:
    """``[(points scanned, edges so far, points searched again exactly), ...]``
    per Boruvka round of the last mr_mst call."""
    L = _load()
    a = (ctypes.c_int64 * 64)()
    e = (ctypes.c_int64 * 64)()
    x = (ctypes.c_int64 * 64)()
    r = L.hdbmst_last_mst_rounds(a, e, x, 64)
    return [(int(a[i]), int(e[i]), int(x[i])) for i in range(min(r, 64))]


def last_knn_exact_rows() -> int:
    """Rows of the last k-NN / core-distance call that the rounding proof left
    open and that were searched exactly over all points."""
    return int(_load().hdbmst_last_knn_exact_rows())


def last_knn_tile_pairs() -> int:
    """(row, column) pairs the distance tile of the last k-NN / core-distance
    call evaluated, in whole 128 x 128 blocks (pruned blocks excluded)."""
    return int(_load().hdbmst_last_knn_tile_pairs())


def last_mst_scan_pairs() -> int:
    """(row, column) pairs the Boruvka scan tiles of the last mr_mst call
    evaluated, over all rounds."""
    return int(_load().hdbmst_last_mst_scan_pairs())


def profile_read() -> dict:
    """Per-kernel ``{name: (total_ms, launches)}`` since the last read; clears the record."""
    L = _load()
    ms = (ctypes.c_double * 64)()
    cnt = (ctypes.c_int64 * 64)()
    nk = L.hdbmst_profile_read(ms, cnt, 64)
    out = {}
    for i in range(nk):
        if cnt[i]:
            out[L.hdbmst_profile_kernel_name(i).decode()] = (ms[i], int(cnt[i]))
    return out
