"""Builds libmgg.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Usage: ``python -m moe_grouped_gemm_persistent_gb300.build [--force] [--verbose] [--checked]``.
The translation units compile in parallel; the CUDA runtime is linked statically, so
the library loads on a machine without a GPU driver (calls then report no device).

``--checked`` builds the bounds-checked variant ``libmgg_checked.so`` (-DMGG_CHECKED): the
kernels test every computed global index, tensor-map slot and TMEM column against the call's
extents and report MGG_ERR_DEVICE_BOUNDS instead of making the access.  It is a debugging
build (slower), loaded instead of ``libmgg.so`` when MGG_LIB_VARIANT=checked.
"""
from __future__ import annotations

import argparse
import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmgg.so")
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB = os.path.join(PKG, "libmgg_checked.so")
SOURCES = ["mgg_api.cu", "dglu_bwd.cu", "wgrad.cu", "wgrad_noalloc.cu", "mgg_testing.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    lib, build_dir = (CHECKED_LIB, CHECKED_BUILD_DIR) if checked else (LIB, BUILD_DIR)
    if checked:
        extra_flags = (*extra_flags, "-DMGG_CHECKED")
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *CFLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print register / shared-memory usage")
    ap.add_argument("--checked", action="store_true", help="build the bounds-checked libmgg_checked.so")
    args = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if args.ptxas_info else []
    print(build(force=args.force or args.ptxas_info, verbose=args.verbose or args.ptxas_info, extra_flags=extra,
                checked=args.checked))


if __name__ == "__main__":
    sys.exit(main())
