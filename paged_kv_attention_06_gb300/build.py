"""Builds libpagedattn.so in-tree with nvcc for sm_103a.

Every .cu file under csrc/ is compiled in parallel (one -gencode, no other
architecture), then linked into ``_build/libpagedattn.so`` against the shared
CUDA runtime. Re-running is cheap: nothing is rebuilt when the library is
newer than every source and header.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(BUILD, "libpagedattn.so")
ROOT = os.path.dirname(HERE)
BENCH_SRC = os.path.join(ROOT, "bench_loop.cpp")
BENCH_LIB = os.path.join(BUILD, "libpabench.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-cudart", "shared",
                     "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.h")) +
            glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) +
            [os.path.abspath(__file__)])


def up_to_date() -> bool:
    for lib in (LIB, BENCH_LIB):
        if not os.path.exists(lib):
            return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(BENCH_LIB))
    return all(os.path.getmtime(p) <= t for p in _deps() + [BENCH_SRC])


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link; returns the library path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or ptxas_info or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}")
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-soname=libpagedattn.so", "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    # The benchmark's native step loops (bench_loop.cpp, beside bench.py):
    # host code only, linked against the library above.
    if os.path.exists(BENCH_SRC):
        tmp = BENCH_LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, "-shared", "-std=c++17", "-O2", "-Xcompiler", "-fPIC", "-cudart", "shared",
               "-I", ROOT, BENCH_SRC, "-o", tmp, "-L", BUILD, "-lpagedattn",
               "-Xlinker", "-rpath=$ORIGIN", "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("bench loop build failed")
        os.replace(tmp, BENCH_LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
