"""Build ``_build/libfv.so`` (the C-ABI library) from ``csrc/`` with nvcc for
sm_103a.  Translation units compile in parallel; rebuilt only when a source
or header is newer than the library."""
from __future__ import annotations

import concurrent.futures
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libfv.so")
# the debug build: the same sources with the in-kernel index checks compiled in
DEBUG_LIB = os.path.join(OUT_DIR, "libfv_debug.so")
DEBUG_FLAGS = ["-DFV_DEBUG_CHECKS=1"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool, debug: bool = False) -> str:
    obj = os.path.join(OUT_DIR, os.path.basename(src) + (".debug.o" if debug else ".o"))
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + (DEBUG_FLAGS if debug else []) + \
        (["-Xptxas", "-v"] if verbose_ptxas else []) + ["-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas:
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Build libfv.so (or, with debug, libfv_debug.so) if a source is newer."""
    lib = DEBUG_LIB if debug else LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and not _stale(lib):
        return lib
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(sources())) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, debug), sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """The release and the debug library, compiled side by side."""
    with concurrent.futures.ThreadPoolExecutor(max_workers=2) as ex:
        list(ex.map(lambda d: build(force=force, debug=d), (False, True)))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
