"""The C ABI from plain C: tests/c_abi/abi_main.c includes only ccl.h and the
CUDA runtime, and links only libccl.so and libcudart.  On the CPU the
program must compile as strict C99 against the header and link against
the library; on a GPU it runs and checks AllReduce, ReduceScatter and
AllGather results and error statuses itself (exit status 0)."""
import glob
import os
import shutil
import subprocess

import pytest

from conftest import ROOT
from reducescatter_reduction_gb300 import build as ccl_build

SRC = os.path.join(ROOT, "tests", "c_abi", "abi_main.c")
OUT = os.path.join(ROOT, "tests", "c_abi", "_build", "abi_main")
PKG = os.path.join(ROOT, "reducescatter_reduction_gb300")


def cuda_paths():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    libs = [d for d in [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets", "*", "lib"))
            if os.path.exists(os.path.join(d, "libcudart.so"))]
    return os.path.join(home, "include"), libs[0]


def compile_program():
    ccl_build.build()
    inc, lib = cuda_paths()
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    # the header alone is strict ISO C99 (CUDA's own headers are not, so the
    # program below is built without -pedantic)
    subprocess.run(["gcc", "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror", "-fsyntax-only", "-x", "c",
                    "-I", os.path.join(ROOT, "include"), "-"], input='#include "ccl.h"\n', check=True,
                   capture_output=True, text=True)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           "-I", os.path.join(ROOT, "include"), "-I", inc, SRC, "-o", OUT,
           "-L", PKG, "-lccl", "-L", lib, "-lcudart",
           "-Wl,-rpath," + PKG, "-Wl,-rpath," + lib]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return OUT


@pytest.mark.cpu
def test_c_program_compiles_as_c99_and_links():
    exe = compile_program()
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
def test_c_program_runs_its_checks():
    exe = compile_program()
    res = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "ok: 0 failure(s)" in res.stdout
