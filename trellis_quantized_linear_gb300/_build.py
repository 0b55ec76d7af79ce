"""Builds libexl3.so in-tree with nvcc for sm_103a (no torch involvement).

Each translation unit is compiled in parallel; objects go to
``trellis_quantized_linear_gb300/_build/`` and the shared library to
``trellis_quantized_linear_gb300/libexl3.so``. With ``bounds_checked`` the
same sources are compiled with ``EXL3_DEBUG_BOUNDS=1`` (every kernel access
checked against its launch's extents) into ``_build_bounds/`` and
``libexl3_bounds.so``. A rebuild happens only when a source or header is
newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libexl3.so")
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(PKG, "libexl3_bounds.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libexl3")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(ROOT, "include", "exl3.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, bounds_checked: bool = False) -> str:
    lib, build_dir = (LIB_BOUNDS, BUILD_BOUNDS) if bounds_checked else (LIB, BUILD)
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    common = [nvcc, "-std=c++17", ARCH, "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
              "-I", os.path.join(ROOT, "include")]
    if bounds_checked:
        common += ["-DEXL3_DEBUG_BOUNDS=1"]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src).replace(".cu", ".o"))
        r = subprocess.run(common + ["-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, ARCH, "-shared", "-o", tmp] + objs + ["-lcudart_static", "-lrt", "-ldl", "-lpthread"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, bounds_checked="--bounds" in sys.argv))
