"""hdbmst_knn_noalloc: k-NN for callers that may not allocate device memory.

Some callers cannot call cudaMalloc or pass a workspace (a host application
that pre-reserved all device memory and gives plugins no allocator, a
latency-critical loop where an allocation could synchronise the device, a
process under a hard memory quota).  This entry point takes its scratch from
a fixed array in the library's device image.  These tests call it through the
C ABI and require the same results as hdbmst_knn, call after call, since every
call reuses the same array and must not depend on what the previous call left
there.  The file is named to be collected last.
"""

import ctypes

import numpy as np
import pytest

import workloads

NOALLOC_BYTES = 64 << 20
ERR_TOO_LARGE = 7


def _lib():
    from hdbscan_mst_gb300 import build
    build.build()
    import hdbscan_mst_gb300 as H
    L = H.lib()
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    L.hdbmst_knn_noalloc.argtypes = [vp, i64, i64, vp, i64, i64, i32, i32, vp, vp, vp]
    L.hdbmst_knn_noalloc.restype = i32
    return H, L


def _noalloc(L, X, Y, k):
    import torch
    d, n = X.shape
    m = Y.shape[1]
    idx = torch.full((n, k), -1, dtype=torch.int32, device="cuda")
    dist = torch.full((n, k), -1.0, dtype=torch.float32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = L.hdbmst_knn_noalloc(X.data_ptr(), X.stride(0), n, Y.data_ptr(), Y.stride(0), m, d, k,
                              idx.data_ptr(), dist.data_ptr(), stream)
    torch.cuda.synchronize()
    return st, idx.cpu().numpy(), dist.cpu().numpy()


@pytest.mark.gpu
def test_noalloc_matches_knn_on_consecutive_calls():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required")
    H, L = _lib()
    # A: 25 000 x 192 against itself fills most of the scratch with the packed
    #    copies (58 MB of the 64 MiB), so the rows go through the candidate
    #    lists in many small chunks.
    XA = workloads.small(25000, 192, seed=21, dup_frac=0.01)
    # B: the 1 416 x 102 section against every 5th point.
    XB, task = workloads.workload("knn_1416_d102")
    YB = workloads.subset_columns(XB, task["y_stride"])
    a = torch.from_numpy(XA).cuda()
    b = torch.from_numpy(XB).cuda()
    yb = torch.from_numpy(YB).cuda()
    ref_a = [t.cpu().numpy() for t in H.knn(a, a, 10)]
    ref_b = [t.cpu().numpy() for t in H.knn(b, yb, 10)]
    for X, Y, ref in ((a, a, ref_a), (b, yb, ref_b), (a, a, ref_a)):
        st, gi, gd = _noalloc(L, X, Y, 10)
        assert st == 0, L.hdbmst_status_string(st)
        # both entry points return the exact k nearest under the library's
        # one distance function, with the same tie order: identical bits
        assert np.array_equal(gi, ref[0])
        assert np.array_equal(gd, ref[1])


def test_noalloc_rejects_problems_beyond_its_scratch():
    """Checked on the host before any GPU work: 100 000 x 192 needs about 230 MB."""
    H, L = _lib()
    vp = ctypes.c_void_p
    st = L.hdbmst_knn_noalloc(vp(256), 100000, 100000, vp(256), 100000, 100000, 192, 10,
                              vp(256), vp(256), None)
    assert st == ERR_TOO_LARGE
    assert b"fixed scratch" in L.hdbmst_status_string(st)
