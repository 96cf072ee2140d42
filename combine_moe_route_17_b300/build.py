"""Builds the CUDA library libmoe_route.so in-tree for sm_103a (B300).

    python -m combine_moe_route_17_b300.build [--force] [--verbose-ptxas]

Each csrc/*.cu compiles to an object under _build/ (rebuilt when it or a
header is newer), then nvcc links them into lib/libmoe_route.so against the
shared CUDA runtime, so the library joins the runtime PyTorch has loaded.
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmoe_route.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    os.makedirs(BUILD, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    hdr_time = max((os.path.getmtime(h) for h in headers()), default=0.0)
    objs = []
    changed = force or not os.path.exists(LIB)
    jobs = []
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if (force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src),
                                                                              hdr_time)):
            tmp = obj + f".tmp{os.getpid()}"
            cmd = [_nvcc(), *NVCC_FLAGS, "-c", src, "-o", tmp]
            if ptxas_verbose:
                cmd[1:1] = ["-Xptxas", "-v"]
            if not quiet:
                print(" ".join(cmd), flush=True)
            jobs.append((cmd, tmp, obj))
    if jobs:
        # the translation units are independent: compile them side by side
        from concurrent.futures import ThreadPoolExecutor

        def compile_one(job):
            cmd, tmp, obj = job
            subprocess.check_call(cmd)
            os.replace(tmp, obj)

        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for fut in [ex.submit(compile_one, j) for j in jobs]:
                fut.result()
        changed = True
    if changed or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
        if not quiet:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    a = ap.parse_args(argv)
    print(build(force=a.force, ptxas_verbose=a.verbose_ptxas, quiet=False))


if __name__ == "__main__":
    sys.exit(main())
