"""Build libdsa.so in-tree for sm_103a with nvcc (one translation unit per
process, compiled in parallel, then linked as a shared library).

build(debug=True) makes libdsa_debug.so instead: the same sources with
-DDSA_DEBUG_BOUNDS, whose kernels check the rows their index-driven gathers
compute and report a row outside its array in the workspace status word.

Usage: python -m top_sparse_attention_chunked_gb300.build_lib [--verbose] [--debug]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdsa.so")
DEBUG_BUILD = os.path.join(HERE, "_build_debug")
DEBUG_LIB = os.path.join(HERE, "libdsa_debug.so")
SOURCES = ["dsa_api.cu", "indexer.cu", "topk.cu", "attention.cu", "prefill_attn.cu",
           "topk_noalloc.cu", "cache_append.cu", "rmsnorm_rotary.cu",
           "rope_append.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    cand = [os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"]
    for c in cand:
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found (needed to build libdsa)")


def _compile(nvcc: str, src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(DEBUG_BUILD if debug else BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           *(["-DDSA_DEBUG_BOUNDS"] if debug else []),
           "-I", os.path.join(HERE, "..", "include"), "-c", os.path.join(CSRC, src),
           "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "dsa.h"))
    return any(os.path.getmtime(f) > t for f in files)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile and link libdsa.so (with `debug`: libdsa_debug.so) unless it is
    newer than every source."""
    lib = DEBUG_LIB if debug else LIB
    if not force and not _stale(lib):
        return lib
    nvcc = nvcc_path()
    os.makedirs(DEBUG_BUILD if debug else BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, verbose, debug), SOURCES))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv, debug="--debug" in sys.argv))
