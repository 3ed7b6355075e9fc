"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, and answers host-side queries (no kernel runs here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hdbmst.h")


@pytest.fixture(scope="module")
def L():
    from hdbscan_mst_gb300 import build
    build.build()
    import hdbscan_mst_gb300 as H
    return H.lib()


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hdbmst_[a-z_]+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared()
    for n in ("hdbmst_knn", "hdbmst_core_distances", "hdbmst_mr_mst", "hdbmst_workspace_bytes",
              "hdbmst_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for name in declared():
        assert hasattr(L, name), f"{name} declared in include/hdbmst.h but not exported"


def test_status_strings(L):
    for s in range(7):
        assert L.hdbmst_status_string(s)
    assert L.hdbmst_status_string(0) == b"ok"


def test_workspace_sizes(L):
    OP_KNN, OP_CORE, OP_MST = 0, 1, 2
    assert L.hdbmst_workspace_bytes(OP_KNN, 1000, 200, 61, 10) > 0
    assert L.hdbmst_workspace_bytes(OP_CORE, 1000, 0, 61, 10) > 0
    assert L.hdbmst_workspace_bytes(OP_MST, 1000, 0, 61, 11) > 0
    assert L.hdbmst_workspace_bytes(OP_MST, 1000, 0, 61, 0) > 0
    # invalid or unsupported sizes give 0
    assert L.hdbmst_workspace_bytes(OP_KNN, 1000, 200, 0, 10) == 0
    assert L.hdbmst_workspace_bytes(OP_KNN, 1000, 200, 61, 33) == 0
    assert L.hdbmst_workspace_bytes(OP_CORE, 10, 0, 61, 11) == 0
    assert L.hdbmst_workspace_bytes(OP_CORE, 1000, 0, 61, 32) == 0
    assert L.hdbmst_workspace_bytes(7, 1000, 0, 61, 1) == 0
    # grows with n
    assert L.hdbmst_workspace_bytes(OP_MST, 200000, 0, 61, 11) > L.hdbmst_workspace_bytes(OP_MST, 2000, 0, 61, 11)


def test_argument_errors_need_no_gpu(L):
    """Host-side validation returns before any CUDA call."""
    vp = ctypes.c_void_p
    # k > m
    assert L.hdbmst_knn(vp(16), 10, 10, vp(16), 5, 5, 3, 6, vp(16), vp(16), vp(256), 1 << 20, None) == 1
    # k beyond the build's limit
    assert L.hdbmst_knn(vp(16), 100, 100, vp(16), 100, 100, 3, 33, vp(16), vp(16), vp(256), 1 << 20, None) == 2
    # d = 0, ld < n
    assert L.hdbmst_knn(vp(16), 10, 10, vp(16), 10, 10, 0, 1, vp(16), vp(16), vp(256), 1 << 20, None) == 1
    assert L.hdbmst_knn(vp(16), 5, 10, vp(16), 10, 10, 3, 1, vp(16), vp(16), vp(256), 1 << 20, None) == 1
    # null outputs
    assert L.hdbmst_knn(vp(16), 10, 10, vp(16), 10, 10, 3, 1, None, vp(16), vp(256), 1 << 20, None) == 1
    # workspace too small / misaligned
    assert L.hdbmst_knn(vp(16), 10, 10, vp(16), 10, 10, 3, 1, vp(16), vp(16), vp(256), 16, None) == 3
    assert L.hdbmst_knn(vp(16), 10, 10, vp(16), 10, 10, 3, 1, vp(16), vp(16), vp(100), 1 << 30, None) == 3
    # an empty query set is valid and does nothing
    assert L.hdbmst_knn(vp(16), 0, 0, vp(16), 10, 10, 3, 1, vp(16), vp(16), None, 0, None) == 0
    # min_samples > n, min_samples + 1 > KMAX
    assert L.hdbmst_core_distances(vp(16), 5, 5, 3, 6, vp(16), None, None, vp(256), 1 << 20, None) == 1
    assert L.hdbmst_core_distances(vp(16), 100, 100, 3, 32, vp(16), None, None, vp(256), 1 << 20, None) == 2
    # one list pointer without the other
    assert L.hdbmst_core_distances(vp(16), 100, 100, 3, 5, vp(16), vp(16), None, vp(256), 1 << 20, None) == 1
    assert L.hdbmst_mr_mst(vp(16), 100, 100, 3, vp(16), vp(16), None, 6, vp(16), vp(16), vp(256), 1 << 20, None) == 1
    # list longer than n
    assert L.hdbmst_mr_mst(vp(16), 10, 10, 3, vp(16), vp(16), vp(16), 11, vp(16), vp(16), vp(256), 1 << 20, None) == 1
    # n <= 1: nothing to do
    assert L.hdbmst_mr_mst(vp(16), 1, 1, 3, vp(16), None, None, 0, None, None, None, 0, None) == 0
    assert L.hdbmst_mr_mst(vp(16), 0, 0, 3, vp(16), None, None, 0, None, None, None, 0, None) == 0


def test_python_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import hdbscan_mst_gb300 as H
    monkeypatch.setattr(H, "_lib", None)
    monkeypatch.setattr(H._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(H.HdbmstUnavailable):
        H.knn(__import__("numpy").zeros((2, 3), "float32"), __import__("numpy").zeros((2, 3), "float32"), 1)


def test_no_oracle_in_product_path():
    """The package never imports the oracle or the test helpers."""
    pkg = os.path.join(ROOT, "hdbscan_mst_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle." not in text.replace("oracle.c", ""), f


def test_mst_workspace_holds_the_pruning_buffers(L):
    """With nearest lists, at most 64 features and at least 16 384 points the
    MST workspace also holds the symmetric scan's pruning buffers: the pivot
    distances of every point (n x 128 floats) and the block-pair bounds and
    lists (blocks^2 each).  Without lists, with wider rows or fewer points it
    does not."""
    OP_MST = 2
    n = 20000
    blocks = (n + 127) // 128
    with_lists = L.hdbmst_workspace_bytes(OP_MST, n, 0, 61, 11)
    without = L.hdbmst_workspace_bytes(OP_MST, n, 0, 61, 0)
    extra = with_lists - without
    assert extra >= n * 128 * 4 + 2 * blocks * blocks * 4
    # 65 features: no tensor-core scan, no pruning buffers (only the lists' own needs differ)
    wide_extra = (L.hdbmst_workspace_bytes(OP_MST, n, 0, 65, 11)
                  - L.hdbmst_workspace_bytes(OP_MST, n, 0, 65, 0))
    assert wide_extra < n * 128 * 4
    small_extra = (L.hdbmst_workspace_bytes(OP_MST, 16000, 0, 61, 11)
                   - L.hdbmst_workspace_bytes(OP_MST, 16000, 0, 61, 0))
    assert small_extra < 16000 * 128 * 4
