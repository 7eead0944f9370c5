"""Build the C-ABI library in-tree for sm_103a with nvcc.

Two variants of the same sources:
  libcpa.so          the library;
  libcpa_checked.so  a checked build for tests (-DCPA_BOUNDS_CHECK: every
                     global index the kernels compute is range-checked and an
                     index out of range sets CPA_EBIT_BOUNDS instead of being
                     used; -DCPA_TEST_HOOKS: a short in-kernel wait limit and a
                     test hook that withholds one tile copy, so that a bounded
                     wait can be made to run out).
Every .cu file of both variants compiles in parallel into _build/<variant>/,
then one link step per variant writes the library next to this file.  A
variant is rebuilt only when a source or header is newer than its library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libcpa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         f"-I{os.path.join(ROOT, 'include')}"]
VARIANTS = {
    "default": ("libcpa.so", []),
    "checked": ("libcpa_checked.so", ["-DCPA_BOUNDS_CHECK", "-DCPA_TEST_HOOKS"]),
}


def lib_file(variant: str = "default") -> str:
    return os.path.join(HERE, VARIANTS[variant][0])


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libcpa.so")
    return path


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))) + \
        [os.path.join(ROOT, "include", "cpa.h"), os.path.abspath(__file__)]


def up_to_date(variant: str = "default") -> bool:
    lib = lib_file(variant)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra=(), variants=("default", "checked")) -> str:
    """Build the requested variants (all by default); returns the path of libcpa.so."""
    todo = [v for v in variants if force or not up_to_date(v)]
    if not todo:
        return LIB
    cc = nvcc()

    def compile_one(job):
        variant, src = job
        out_dir = os.path.join(BUILD, variant)
        os.makedirs(out_dir, exist_ok=True)
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *FLAGS, *VARIANTS[variant][1], *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({variant}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return variant, obj

    jobs = [(v, s) for v in todo for s in _sources()]
    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, jobs))
    for v in todo:
        lib = lib_file(v)
        tmp = lib + ".tmp"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *[o for vv, o in objs if vv == v]],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed ({v}):\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if v else []
    print(build(force=True, verbose=v, extra=extra))
