"""Build the C-ABI shared library libpa_gb300.so in-tree (sm_103a only).

    python paged_kv_cache_161_gb300/build.py [--force] [--verbose] [--ptxas]

(run as a script: importing the package itself requires the built library)

Each CUDA translation unit is compiled by nvcc in parallel, the host units by g++, and
nvcc links them with the static CUDA runtime, so the library needs only the driver at
run time (and loads, without calling into CUDA, on a machine with no GPU).
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libpa_gb300.so")

CU_SOURCES = ["errors.cu", "kv_write.cu", "copy_blocks.cu", "decode_attention.cu", "decode_mma.cu", "prefill_attention.cu",
              "attention_fixed_scratch.cu", "prefill_tcgen05.cu"]
CPP_SOURCES = ["api.cpp", "block_manager.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _cuda_home() -> str:
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "bin", "nvcc")):
            return c
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found: set CUDA_HOME")


def _headers():
    hs = [os.path.join(INCLUDE, "pa.h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(p) > t for p in [src] + _headers())


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed ({r.returncode}):\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (what changed) and link; returns the library path."""
    cuda = _cuda_home()
    nvcc = os.path.join(cuda, "bin", "nvcc")
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    jobs, objs = [], []
    for f in CU_SOURCES:
        src, obj = os.path.join(CSRC, f), os.path.join(BUILD_DIR, f + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            cmd = [nvcc, *ARCH, "-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "-c", src, "-o", obj]
            if ptxas_verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)
    cxx = os.environ.get("CXX", "g++")
    for f in CPP_SOURCES:
        src, obj = os.path.join(CSRC, f), os.path.join(BUILD_DIR, f + ".o")
        objs.append(obj)
        if force or _stale(obj, src):
            jobs.append([cxx, "-std=c++17", "-O2", "-fPIC", "-Wall", "-I", INCLUDE, "-I",
                         os.path.join(cuda, "include"), "-c", src, "-o", obj])
    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            list(ex.map(lambda c: _run(c, verbose), jobs))
    if jobs or not os.path.exists(LIB_PATH):
        tmp = LIB_PATH + ".tmp"
        _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], verbose)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas", action="store_true", help="print register / spill / smem use")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas))


if __name__ == "__main__":
    sys.exit(main())
