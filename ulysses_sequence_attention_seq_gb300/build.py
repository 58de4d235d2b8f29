"""Builds libulysses.so in-tree with nvcc for sm_103a (no cmake, no setuptools).

Every .cu file under csrc/ is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically, so the library loads on a
machine without a GPU (the host-only entry points then still work).

build(checked=True) builds the range-checked variant (-DULYSSES_CHECK_BOUNDS:
every plain global load and store is checked against its buffer, see
csrc/check.cuh) into _build_checked/; select it with ULYSSES_LIB.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libulysses.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libulysses.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    extra = ["-DULYSSES_CHECK_BOUNDS"] if checked else []
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                     glob.glob(os.path.join(INCLUDE, "*.h")))
    nvcc = _nvcc()
    procs, objs = [], []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            cmd = [nvcc, *ARCH, *FLAGS, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
            log = open(obj + ".log", "w")
            procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, pr, log in procs:
        pr.wait()
        log.close()
        if pr.returncode != 0:
            failed.append(src)
        if verbose or pr.returncode != 0:
            sys.stderr.write(open(log.name).read())
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f) for f in failed))
    if force or _stale(lib, objs):
        tmp = lib + f".{os.getpid()}.tmp"
        subprocess.check_call([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
