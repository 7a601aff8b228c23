"""Builds libcsa_index.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG, "libcsa_index.so")
SOURCES = [os.path.join(CSRC, f) for f in ("csa_index.cu", "csa_writer.cu", "csa_recall.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("csa_ptx.cuh", "csa_select.cuh", "csa_score64.cuh",
                                                  "csa_internal.h")] + [
    os.path.join(INCLUDE, "csa_index.h")]
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH") or "/usr/local/cuda"
    cand = os.path.join(home, "bin", "nvcc")
    if os.path.exists(cand):
        return cand
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the library unless it is newer than every source. Returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           f"-I{INCLUDE}", "-o", tmp] + SOURCES
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


# Test builds: the same sources with compile-time switches that only tests use
# (for example a short pipeline wait limit and a delayed producer, to exercise
# the bounded-wait path). Each goes to its own file next to the product library.
TEST_VARIANTS = {
    "timeout": ["-DCSA_TEST_WAIT_LIMIT_NS=20000ull", "-DCSA_TEST_WALKER_DELAY_NS=200000ull"],
}


def build_test_variant(name: str, force: bool = False) -> str:
    """Compiles test variant `name` (see TEST_VARIANTS) unless up to date. Returns its path."""
    path = os.path.join(PKG, f"libcsa_index_test_{name}.so")
    if not force and os.path.exists(path) and all(os.path.getmtime(d) <= os.path.getmtime(path) for d in DEPS):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = [nvcc_path(), ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           f"-I{INCLUDE}", "-o", tmp] + TEST_VARIANTS[name] + SOURCES
    subprocess.run(cmd, check=True)
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
