"""Builds the in-tree CUDA library ``_build/libep_gb300.so`` for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically. The library exports
the C ABI of ``include/ep.h``. ``--checked`` builds the checked variant
``_build/libep_gb300_checked.so`` instead (EP_CHECKED=1: every kernel access
tested against its buffer; same ABI plus the test hook
``ep_checked_trim_extent``).

    python -m combine_topk_ids_dest_gb300.build [--force] [--verbose] [--checked]
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libep_gb300.so")
LIB_CHECKED = os.path.join(BUILD, "libep_gb300_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE fp32 everywhere: no flush-to-zero, no contraction of separate adds/multiplies.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-Wall,-Wextra", "-ftz=false",
              "-prec-div=true", "-prec-sqrt=true", "-fmad=false", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libep_gb300.so")


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile (when sources are newer than the library) and return its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and not _stale(lib):
        return lib
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + (["-DEP_CHECKED=1"] if checked else []) + list(extra_flags) + \
        (["-Xptxas", "-v"] if verbose else [])

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, checked=args.checked))
