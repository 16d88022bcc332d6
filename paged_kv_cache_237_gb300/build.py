"""Build the C-ABI library ``libpa_gb300.so`` in-tree for sm_103a.

nvcc compiles each CUDA translation unit with
``-gencode arch=compute_103a,code=sm_103a -O3 -lineinfo``; the host block
manager and ABI glue go through g++.  The CUDA runtime is linked statically,
so the library loads without a GPU (compute calls then fail with PA_ERR_CUDA).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libpa_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CUDA_SOURCES = ["pa_decode.cu", "pa_decode_simt.cu", "pa_cache.cu"]
CXX_SOURCES = ["block_manager.cpp", "pa_api.cpp"]
HEADERS = ["pa_internal.h", "pa_decode_common.cuh"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    srcs = [os.path.join(CSRC, f) for f in CUDA_SOURCES + CXX_SOURCES + HEADERS]
    return srcs + [os.path.join(INCLUDE, "pa.h"), os.path.abspath(__file__)]


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library.  Several
    processes may call this at once (one per rank): a file lock lets one of
    them compile while the others wait and then find the library fresh."""
    if not force and not _stale(LIB_PATH):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    import fcntl
    with open(os.path.join(BUILD_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and not _stale(LIB_PATH):
                return LIB_PATH
            return _compile(verbose, ptxas_verbose)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _compile(verbose: bool, ptxas_verbose: bool) -> str:
    nvcc = _nvcc()
    common = ["-std=c++17", "-O3", f"-I{INCLUDE}", f"-I{CSRC}"]
    jobs = []
    for f in CUDA_SOURCES:
        obj = os.path.join(BUILD_DIR, f + ".o")
        cmd = [nvcc, *ARCH, *common, "-lineinfo", "-Xcompiler", "-fPIC", "-c",
               os.path.join(CSRC, f), "-o", obj]
        if ptxas_verbose:
            cmd += ["-Xptxas", "-v"]
        jobs.append((cmd, obj))
    for f in CXX_SOURCES:
        obj = os.path.join(BUILD_DIR, f + ".o")
        cmd = ["g++", *common, "-fPIC", "-Wall", "-c", os.path.join(CSRC, f), "-o", obj]
        jobs.append((cmd, obj))

    def run(job):
        cmd, _ = job
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(run, jobs))
    for cmd, r in results:
        if verbose or ptxas_verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {cmd[-3]}")
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-lpthread", "-ldl"]
    r = subprocess.run(link, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(" ".join(link) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError("link failed")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="--ptxas" in sys.argv))
