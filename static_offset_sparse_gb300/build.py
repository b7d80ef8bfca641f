"""Build libsfa.so in-tree for sm_103a with nvcc (no cmake).

Usage: ``python -m static_offset_sparse_gb300.build`` or ``build()``.
Each translation unit compiles in its own process; the link step writes
``static_offset_sparse_gb300/libsfa.so`` next to this file.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsfa.so")

DEBUG_LIB = os.path.join(PKG, "libsfa_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["sfa_host.cpp", "sfa_api.cu", "sfa_fwd.cu", "sfa_bwd.cu", "sfa_fwd_tc.cu", "sfa_bwd_tc.cu",
           "sfa_noalloc.cu", "sfa_decode.cu", "sfa_schedule.cpp", "sfa_band.cu"]
# The bounds-checked build (libsfa_debug.so) recompiles the SIMT kernels with
# SFA_DEBUG_BOUNDS: every row index they form is range-checked, a bad one is
# recorded as SFA_ERR_DEVICE_BOUNDS and its access skipped.
DEBUG_SOURCES = ["sfa_fwd.cu", "sfa_bwd.cu"]


def _nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsfa")
    return p


def _compile(src: str, verbose: bool, debug_bounds: bool = False) -> str:
    obj = os.path.join(OUT, ("dbg_" if debug_bounds else "") + os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), "-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2",
           "-I", os.path.join(ROOT, "include"), "-I", CSRC, "-c", os.path.join(CSRC, src), "-o", obj]
    if debug_bounds:
        cmd.insert(1, "-DSFA_DEBUG_BOUNDS")
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "c++"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def _link(objs, lib: str) -> None:
    tmp = lib + ".tmp"
    cmd = [_nvcc(), "-shared", *ARCH, "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(verbose: bool = False, debug_bounds: bool = True) -> str:
    """Compile every source for sm_103a and link libsfa.so (and, with
    debug_bounds, the bounds-checked libsfa_debug.so); returns libsfa.so's path."""
    os.makedirs(OUT, exist_ok=True)
    jobs = [(s, False) for s in SOURCES] + ([(s, True) for s in DEBUG_SOURCES] if debug_bounds else [])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], verbose, j[1]), jobs))
    main = objs[:len(SOURCES)]
    _link(main, LIB)
    if debug_bounds:
        dbg = dict(zip(DEBUG_SOURCES, objs[len(SOURCES):]))
        _link([dbg.get(s, o) for s, o in zip(SOURCES, main)], DEBUG_LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
