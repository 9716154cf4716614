"""Builds libswa.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m sink_sparse_attention_swa_b300.build [--verbose-ptxas] [--debug]

Each .cu under csrc/ is compiled in parallel to an object under _build/, then
linked into sink_sparse_attention_swa_b300/libswa.so against the shared CUDA
runtime (so that the current device and streams are the ones torch uses).
With --debug (build(debug=True)) the same sources are compiled with SWA_DEBUG
defined, under _build_debug/, into libswa_debug.so: the kernels' bounds checks
are compiled in (see include/swa.h).
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libswa.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libswa_debug.so")
INCLUDE = os.path.join(ROOT, "include")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-Wall", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(x) > t for x in inputs)


def _compile(src, ptxas_verbose, debug=False):
    obj = os.path.join(BUILD_DEBUG if debug else BUILD, os.path.basename(src)[:-3] + ".o")
    if not _stale(obj, [src] + _deps()) and not ptxas_verbose:
        return obj, ""
    cmd = [NVCC] + ARCH + FLAGS + (["-DSWA_DEBUG"] if debug else []) + (
        ["-Xptxas", "-v"] if ptxas_verbose else []) + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(ptxas_verbose: bool = False, quiet: bool = True, debug: bool = False) -> str:
    out_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose, debug), srcs))
    objs = [o for o, _ in results]
    if ptxas_verbose:
        for _, log in results:
            sys.stderr.write(log)
    if _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs + [
            "-Xlinker", f"-rpath,{CUDA_HOME}/lib64"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    if not quiet:
        print(lib)
    return lib


if __name__ == "__main__":
    build(ptxas_verbose="--verbose-ptxas" in sys.argv, quiet=False, debug="--debug" in sys.argv)
