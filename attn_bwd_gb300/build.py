"""Builds the in-tree CUDA library ``attn_bwd_gb300/libattn_bwd_gb300.so`` for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel with nvcc, then
linked into one shared library exporting the C ABI of ``include/fa.h``.
``--debug-bounds`` builds ``libattn_bwd_gb300_bounds.so`` instead: the same
library compiled with -DFA_DEBUG_BOUNDS, whose kernels check every tile
coordinate and store index against their tensors' extents (FA_ERR_BOUNDS).
Usage:  python -m attn_bwd_gb300.build [--force] [--debug-bounds]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libattn_bwd_gb300.so")
LIB_BOUNDS = os.path.join(PKG, "libattn_bwd_gb300_bounds.so")
SOURCES = ["api.cu", "bwd_main.cu", "bwd_main_persist.cu", "bwd_dq.cu", "bwd_dq_persist.cu", "bwd_aux.cu", "fwd.cu",
           "fwd_persist.cu", "noalloc.cu", "host_pipeline.cu"]
HEADERS = ["kernels.h", "ptx.cuh", "seq.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] +
            [os.path.join(ROOT, "include", "fa.h"), os.path.abspath(__file__)])


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def _compile(src: str, out_dir: str, extra: list[str]) -> tuple[str, str]:
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + FLAGS + extra + ["-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(os.path.join(out_dir, src + ".log"), "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library (the bounds-checking
    debug library with debug_bounds=True)."""
    lib = LIB_BOUNDS if debug_bounds else LIB
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.join(BUILD, "bounds") if debug_bounds else BUILD
    extra = ["-DFA_DEBUG_BOUNDS"] if debug_bounds else []
    os.makedirs(out_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, out_dir, extra), SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
