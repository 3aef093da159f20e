"""Builds the CUDA library libmoe_b300.so in-tree for sm_103a.

    python -m expert_dispatch_top_b300.build [--verbose] [--checked]

Each csrc/*.cu is compiled to an object in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a -O3 -lineinfo), then linked into
expert_dispatch_top_b300/_lib/libmoe_b300.so (static CUDA runtime).  Objects
are rebuilt only when a source or header is newer.  --checked builds the
debugging variant libmoe_b300_checked.so with -DMOE_CHECKED (index range
checks reported in the status word; see moe_build_checked in include/moe.h).
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
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libmoe_b300.so")
LIB_CHECKED = os.path.join(OUT_DIR, "libmoe_b300_checked.so")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", INCLUDE, "-I", CSRC]


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose, build_dir, defines):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    if not _stale(obj, [src] + _headers()):
        return obj, ""
    cmd = [NVCC, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    build_dir = BUILD_DIR + ("_checked" if checked else "")
    defines = ["-DMOE_CHECKED"] if checked else []
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, build_dir, defines), srcs))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            if log:
                print(log, file=sys.stderr)
    if _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, checked="--checked" in sys.argv))
