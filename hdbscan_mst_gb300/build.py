"""Compile the CUDA library ``libhdbmst.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` compiles to an object under ``_build/`` in parallel, then
nvcc links the shared library next to this file.  No cmake: nvcc only.
"""

from __future__ import annotations

import concurrent.futures
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libhdbmst.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the hdbmst CUDA library cannot be built")


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) \
        + [os.path.join(INCLUDE, "hdbmst.h")]
    return srcs, deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    _, deps = _inputs()
    return os.path.getmtime(LIB) >= max(os.path.getmtime(p) for p in deps)


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Build ``libhdbmst.so`` if any source is newer; returns its path."""
    if not force and up_to_date():
        return LIB
    srcs, _ = _inputs()
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = FLAGS + (["-Xptxas", "-v"] if verbose else []) + list(extra or [])

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        r = subprocess.run([cc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, log in results:
            print(log)
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
