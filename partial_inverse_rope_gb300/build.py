"""Build ``libinvrope.so`` in-tree with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into one shared
library next to this file. The CUDA runtime is linked statically; the driver
API (tensor-map encoding) is resolved at run time, so the library loads on a
machine without a GPU driver.
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libinvrope.so")
# debug-bounds variant: device-side index checks that record a fault code
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG, "libinvrope_debug.so")

SOURCES = ["postmix.cu", "remap.cu", "api.cpp", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libinvrope.so")
    return cand


def _common_flags(extra=()):
    return ["-std=c++17", "-O3", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, *extra]


def compile_one(src: str, extra=(), verbose=False, build_dir=BUILD_DIR) -> str:
    os.makedirs(build_dir, exist_ok=True)
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc(), *_common_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cu"):
        cmd[1:1] = [*ARCH, "-lineinfo"]
    else:
        cmd[1:1] = ["-x", "cu", *ARCH]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}")
    return obj


def build(verbose: bool = False, extra=(), debug_bounds: bool = False) -> str:
    """Compile every source for sm_103a and link ``libinvrope.so`` (or, with
    ``debug_bounds``, ``libinvrope_debug.so`` with the device-side index
    checks); returns its path."""
    build_dir, lib_path = (DEBUG_BUILD_DIR, DEBUG_LIB_PATH) if debug_bounds else (BUILD_DIR, LIB_PATH)
    if debug_bounds:
        extra = (*extra, "-DINVROPE_DEBUG_BOUNDS")
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: compile_one(s, extra, verbose, build_dir), SOURCES))
    tmp = lib_path + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or res.returncode != 0:
        sys.stderr.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"linking {os.path.basename(lib_path)} failed")
    os.replace(tmp, lib_path)
    return lib_path


def main():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true", help="print registers / spills / smem")
    ap.add_argument("--debug-bounds", action="store_true",
                    help="build libinvrope_debug.so with device-side index checks")
    args = ap.parse_args()
    extra = ("-Xptxas", "-v") if args.ptxas_info else ()
    print(build(verbose=args.verbose or args.ptxas_info, extra=extra, debug_bounds=args.debug_bounds))


if __name__ == "__main__":
    main()
