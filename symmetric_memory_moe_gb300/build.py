"""Builds libsymm_a2a.so in-tree with nvcc for sm_103a (GB300).

Each .cu file compiles to an object in parallel, then nvcc links the shared
library (CUDA runtime linked statically).  ptxas register/spill reports land
in ``_build/ptxas_<name>.log``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libsymm_a2a.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
SOURCES = ["heap.cu", "a2a.cu", "pc_noalloc.cu", "collectives.cu", "two_phase.cu",
           "ag_gemm.cu", "host_pipe.cu"]
HEADERS = ["symm_device.cuh", "symm_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsymm_a2a.so")


def _inputs() -> list[str]:
    root = os.path.dirname(HERE)
    return ([os.path.join(CSRC, f) for f in SOURCES + HEADERS] +
            [os.path.join(root, "include", "symm_a2a.h"), os.path.abspath(__file__)])


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, defines: tuple = (),
          out: str | None = None) -> str:
    """Compile (if stale) and return the path of libsymm_a2a.so.  `defines`
    (e.g. ("SYMM_PC_UNROLL=8",)) and `out` build a tuning variant elsewhere."""
    if out is None and not defines and not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    lib_path = out or LIB_PATH
    build_dir = os.path.dirname(lib_path) if out else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    dflags = [f"-D{d}" for d in defines]

    def compile_one(src: str) -> str:
        name = os.path.splitext(src)[0]
        obj = os.path.join(build_dir, name + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *dflags, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        with open(os.path.join(build_dir, f"ptxas_{name}.log"), "w") as f:
            f.write(res.stdout + res.stderr)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stderr[-4000:]}")
        if verbose:
            print(res.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stderr[-4000:]}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
