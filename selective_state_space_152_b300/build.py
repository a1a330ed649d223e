"""Build libselscan.so in-tree with nvcc for sm_103a (B300).

    python -m selective_state_space_152_b300.build [--force] [--verbose]

Every ``csrc/*.cu`` file is compiled to an object under ``_build/`` and the
objects are linked into ``selective_state_space_152_b300/libselscan.so``
against the shared CUDA runtime.  No GPU is needed to build.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libselscan.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", f"-I{INCLUDE}", f"-I{CSRC}"]
# Per-file extras.  The chunked kernel's file holds several hundred instantiations: compiling its
# device code in parallel (--split-compile) cuts the clean build from about 8 to 2 minutes.  The split
# build is not deterministic (two builds of one source can differ in register allocation, and the
# row-sequential kernel's time with it), so the files of the kernels that run by default are compiled
# as one unit.
FILE_FLAGS = {"selscan_fwd.cu": ["--split-compile=0"]}


def _nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    hdrs = _headers()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    todo = [(s, o) for s, o in zip(srcs, objs) if force or _stale(o, [s, *hdrs, __file__])]

    def compile_one(so):
        s, o = so
        cmd = [nvcc, *NVCC_FLAGS, *FILE_FLAGS.get(os.path.basename(s), []), *(["-Xptxas", "-v"] if ptxas_info else []),
               "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, cmd, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(todo)))) as ex:
        for s, cmd, r in ex.map(compile_one, todo):
            if verbose or ptxas_info or r.returncode:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode:
                failed.append(s)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if force or todo or _stale(LIB, objs):
        libdir = _cuda_lib_dir(nvcc)
        cmd = [nvcc, "-shared", *ARCH, "-cudart", "shared", *objs, "-o", LIB, "-Xlinker", f"-rpath,{libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("link of libselscan.so failed")
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / shared memory per kernel")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_info=a.ptxas_info))


if __name__ == "__main__":
    main()
