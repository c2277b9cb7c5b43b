"""Builds the HLA-2 CUDA library (libhla2.so) in-tree for sm_103a.

Every translation unit is compiled by nvcc in parallel, then linked into
``chunked_scan_mixer_gb300/_build/libhla2.so``.  Nothing is installed.  ``--debug`` builds
the bounds-checking variant (HLA2_DEBUG: global-memory indices checked against the buffer
extents, a failed check recorded and the access skipped; see hla2_debug_status) into
``chunked_scan_mixer_gb300/_build_debug/libhla2.so``.

    python -m chunked_scan_mixer_gb300.build [--force] [--ptxas-v] [--debug]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libhla2.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libhla2.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the HLA-2 CUDA library cannot be built")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(ROOT, "include", "*.h")))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None, debug: bool = False) -> str:
    nvcc = _nvcc()
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DHLA2_DEBUG"] if debug else [])
    objdir = os.path.join(build_dir, "obj")
    os.makedirs(objdir, exist_ok=True)
    hdrs = _headers()
    srcs = sources()
    objs = []
    todo = []
    for s in srcs:
        o = os.path.join(objdir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + hdrs):
            todo.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [nvcc] + flags + (["-Xptxas", "-v"] if ptxas_verbose else []) + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(s)}:\n{r.stderr}")
        return r.stderr

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for log in ex.map(compile_one, todo):
                if ptxas_verbose and log:
                    sys.stderr.write(log)
    if force or todo or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-v", action="store_true")
    ap.add_argument("--debug", action="store_true", help="the bounds-checking build (HLA2_DEBUG)")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_verbose=args.ptxas_v, debug=args.debug))


if __name__ == "__main__":
    main()
