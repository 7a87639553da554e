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
UNITS = ("msa_indexer.cu", "prefill.cu")  # translation units, compiled in parallel

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


def _common_flags():
    return [*ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def compile_command(unit: str, obj: str, verbose_ptxas: bool = False):
    cmd = [_nvcc(), *_common_flags(), "-c", "-o", obj, os.path.join(CSRC, unit)]
    if verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def link_command(objs, out: str):
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(_nvcc())), "lib64")
    return [_nvcc(), *ARCH_FLAGS, "-shared", "-cudart", "shared", "-Xlinker", f"-rpath={cuda_lib}",
            "-o", out, *objs]


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    """Compile the library if any source is newer than it; returns its path."""
    if not force and not needs_build():
        return LIBRARY
    os.makedirs(LIB_DIR, exist_ok=True)
    from concurrent.futures import ThreadPoolExecutor
    tag = f".tmp{os.getpid()}"
    objs = [os.path.join(LIB_DIR, os.path.splitext(u)[0] + tag + ".o") for u in UNITS]
    try:
        with ThreadPoolExecutor(len(UNITS)) as ex:
            runs = list(ex.map(lambda uo: subprocess.run(compile_command(uo[0], uo[1], verbose_ptxas)),
                               zip(UNITS, objs)))
        for u, r in zip(UNITS, runs):
            if r.returncode != 0:
                raise subprocess.CalledProcessError(r.returncode, f"nvcc {u}")
        tmp = LIBRARY + tag
        subprocess.run(link_command(objs, tmp), check=True)
        os.replace(tmp, LIBRARY)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
