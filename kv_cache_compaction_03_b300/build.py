"""Build libkvc.so (sm_103a) in-tree with nvcc.

Usage: python -m kv_cache_compaction_03_b300.build [--force] [--debug]

--debug builds libkvc_debug.so instead: the same kernels compiled with
KVC_DEBUG, in which the kernels check their indices against the buffers they
were given and record the first bad access in a per-head status word
(KVC_ERR_DEBUG_BOUNDS) instead of performing it.  The binding loads it when
KVC_LIBRARY=debug is set.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libkvc.so")
LIB_DEBUG = os.path.join(PKG, "libkvc_debug.so")
SOURCES = ["kvc_api.cu", "tmap.cu", "attn_tc.cu", "gram_tc.cu", "attn_simt.cu", "select.cu", "gram.cu", "linalg.cu", "sweep.cu", "noalloc.cu", "decode.cu", "omp.cu", "tam.cu", "vconv.cu"]
HEADERS = ["common.cuh", "tc.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "kvc.h")]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every CUDA source into libkvc.so (libkvc_debug.so with debug)
    next to this file; returns its path."""
    lib = LIB_DEBUG if debug else LIB
    if not force and not _stale(lib):
        return lib
    objdir = os.path.join(PKG, "_build_debug" if debug else "_build")
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    extra = list(NVCC_FLAGS) + (["-DKVC_DEBUG=1"] if debug else [])

    def compile_one(s):
        obj = os.path.join(objdir, s.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *extra, "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, s), "-o", obj]
        return s, obj, subprocess.run(cmd, capture_output=True, text=True)

    # the translation units are independent: compile them side by side
    workers = max(1, min(len(SOURCES), os.cpu_count() or 1))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = []
    for s, obj, r in results:
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {s}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        objs.append(obj)
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
