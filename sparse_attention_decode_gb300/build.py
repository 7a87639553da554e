"""Builds libmsa_indexer.so in-tree with nvcc for sm_103a (GB300)."""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(HERE, "_lib")
LIBRARY = os.path.join(LIB_DIR, "libmsa_indexer.so")
MAIN_SOURCE = os.path.join(CSRC, "msa_indexer.cu")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the indexer")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def needs_build(out: str = LIBRARY) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in sources())


def command(out: str = LIBRARY, verbose_ptxas: bool = False):
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(_nvcc())), "lib64")
    cmd = [_nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-shared", "-cudart", "shared", f"-I{INCLUDE}", "-Xlinker", f"-rpath={cuda_lib}",
           "-o", out, MAIN_SOURCE]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the library if any source is newer than it; returns its path."""
    if not force and not needs_build():
        return LIBRARY
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIBRARY + f".tmp{os.getpid()}"
    subprocess.run(command(tmp, verbose_ptxas), check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
