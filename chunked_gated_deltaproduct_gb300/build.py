"""Build step of the CUDA library: every ``csrc/*.cu`` compiled for sm_103a and
linked into ``libgdp_gb300.so`` next to this file (in-tree, git-ignored).  The
debug-bounds variant (``-DGDP_DEBUG_BOUNDS=1``: range checks on the kernels'
descriptor-derived global indices, see the header) links into
``libgdp_gb300_debug.so`` from its own object folder.

Translation units compile in parallel with nvcc; one ``-gencode``
(``arch=compute_103a,code=sm_103a``); no cmake.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdp_gb300.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libgdp_gb300_debug.so")
DEBUG_FLAGS = ["-DGDP_DEBUG_BOUNDS=1"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdp_gb300.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(PKG, "..", "include", "*.h"))


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug_bounds: bool = False) -> str:
    """Compile and link the library (or its debug-bounds variant) if any source is newer than it."""
    lib, folder = (LIB_DEBUG, BUILD_DEBUG) if debug_bounds else (LIB, BUILD)
    extra_flags = [*extra_flags, *(DEBUG_FLAGS if debug_bounds else [])]
    if not force and not is_stale(lib):
        return lib
    os.makedirs(folder, exist_ok=True)
    cc = nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(folder, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys

    flags = sys.argv[1:]
    print(build(force=True, verbose=True, extra_flags=flags))
