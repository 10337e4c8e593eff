"""In-tree build of libgdn_tree.so (nvcc, sm_103a only)."""

from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libgdn_tree.so")
# debug build: every computed global index of the verify, commit and attention kernels checked
# against its array (GDN_STATUS_OUT_OF_BOUNDS, access skipped, no trap)
LIB_DEBUG_BOUNDS = os.path.join(PKG, "libgdn_tree_debug_bounds.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared", "-cudart", "shared",
    "-Xlinker", "-rpath,/usr/local/cuda/lib64",
]


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile every .cu under csrc/ into one shared library, if missing or out of date.
    ``debug_bounds`` builds the address-checking library instead (a separate file)."""
    lib = LIB_DEBUG_BOUNDS if debug_bounds else LIB
    if not force and not stale(lib):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    extra = ["-DGDN_DEBUG_BOUNDS"] if debug_bounds else []
    cmd = [NVCC, *NVCC_FLAGS, *extra, f"-I{INCLUDE}", f"-I{CSRC}", "-o", tmp, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))
