"""Build libccl.so (the C-ABI library) in-tree for sm_103a.

Each source in csrc/ is compiled by its own nvcc process (in parallel); the
objects go to csrc/_build/ and are linked into reducescatter_reduction_gb300/libccl.so.
Sources whose object is newer than the source and every header are skipped.

build_checked() builds the same sources with CCL_BOUNDS_CHECK defined into
csrc/_build/checked/ and libccl_checked.so: every kernel then tests the extent
of each global access it computes against its rank buffer and records a
violation instead of making the access (a test aid; not built by default).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(CSRC, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libccl.so")
BUILD_CHECKED = os.path.join(BUILD, "checked")
LIB_CHECKED = os.path.join(PKG, "libccl_checked.so")
CHECKED_FLAGS = ["-DCCL_BOUNDS_CHECK=1"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libccl.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(CSRC, "*.inc")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _compile(src: str, extra, verbose: bool, build_dir: str = BUILD, cache: bool = True) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    newest_dep = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest_dep and cache:
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj + ".tmp"]
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    if res.stderr.strip() and verbose:
        print(res.stderr, flush=True)
    os.replace(obj + ".tmp", obj)
    return obj


def _build(build_dir: str, lib: str, flags, cache: bool, force: bool, verbose: bool) -> str:
    os.makedirs(build_dir, exist_ok=True)
    if force:
        for o in glob.glob(os.path.join(build_dir, "*.o")):
            os.remove(o)
    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(lambda s: _compile(s, flags, verbose, build_dir, cache), srcs))
    if (not os.path.exists(lib) or force or not cache
            or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs)):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        if verbose:
            print(" ".join(cmd), flush=True)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib)
    return lib


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every csrc/ source and link libccl.so; returns its path."""
    return _build(BUILD, LIB, list(extra_flags), not extra_flags, force, verbose)


def build_checked(force: bool = False, verbose: bool = False) -> str:
    """The checked build (CCL_BOUNDS_CHECK): libccl_checked.so; returns its path."""
    return _build(BUILD_CHECKED, LIB_CHECKED, CHECKED_FLAGS, True, force, verbose)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
