"""Build libdfa.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

Translation units are compiled in parallel into ``_build/`` and linked into
``long_context_flashattention_gb300/libdfa.so``.  A rebuild happens only when a
source or header is newer than the library.

``build(debug_bounds=True)`` (or ``python build.py --debug-bounds``) builds the
bounds-checking variant ``libdfa_bounds.so`` with ``-DDFA_DEBUG_BOUNDS``: the
attention kernels check every global index they compute against its tensor's
extent, skip a violating access and report DFA_ERR_BOUNDS through the status
word.  dfa.py loads it when DFA_DEBUG_BOUNDS=1.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdfa.so")
LIB_BOUNDS = os.path.join(PKG, "libdfa_bounds.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "dfa.h")]


def up_to_date(debug_bounds: bool = False) -> bool:
    lib = LIB_BOUNDS if debug_bounds else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    lib = LIB_BOUNDS if debug_bounds else LIB
    if not force and up_to_date(debug_bounds):
        return lib
    objdir = os.path.join(BUILD, "bounds") if debug_bounds else BUILD
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-DDFA_DEBUG_BOUNDS"] if debug_bounds else []

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                debug_bounds="--debug-bounds" in sys.argv))
