"""Build the CUDA library ``libmsda.so`` in-tree with nvcc for sm_103a.

The library exports the C ABI declared in ``include/msda.h``.  The runtime is
linked statically, so the .so loads on machines without a GPU (only calls
that touch the device need one).  ``build_checked`` builds the same sources
with ``-DMSDA_BOUNDS_CHECK`` into ``libmsda_checked.so``: every data-dependent
row access tests its index and reports a violation through the device error
word instead of making it (for tests; the product loads ``libmsda.so``).
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libmsda.so")
CHECKED_LIB = os.path.join(PKG, "libmsda_checked.so")
SOURCES = ["msda_kernels.cu", "msda_api.cpp", "msda_noalloc.cu"]
HEADERS = ["msda_device.cuh", "msda_forward.cuh", "msda_backward.cuh", "msda_launch.h",
           "msda_linear.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "msda.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB) -> str:
    if not force and not _stale(lib):
        return lib
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-cudart", "static",
           "-I", os.path.join(ROOT, "include"), *extra_flags, "-o", tmp]
    cmd += [os.path.join(CSRC, f) for f in SOURCES]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def build_checked(force: bool = False, verbose: bool = False) -> str:
    return build(force=force, verbose=verbose, extra_flags=("-DMSDA_BOUNDS_CHECK",),
                 lib=CHECKED_LIB)


CEILING_LIB = os.path.join(PKG, "libmsda_ceiling.so")
CEILING_SRC = os.path.join(CSRC, "msda_ceiling.cu")


def build_ceiling(force: bool = False, verbose: bool = False) -> str:
    """The on-chip ceiling probes (a measurement tool, not part of the ABI)."""
    if (not force and os.path.exists(CEILING_LIB)
            and os.path.getmtime(CEILING_LIB) >= os.path.getmtime(CEILING_SRC)):
        return CEILING_LIB
    tmp = CEILING_LIB + ".tmp"
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "-cudart", "static", "-o", tmp, CEILING_SRC]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, CEILING_LIB)
    return CEILING_LIB


if __name__ == "__main__":
    args = sys.argv[1:]
    extra = [a for a in args if a not in ("--force",)]
    print(build(force=True, verbose=True, extra_flags=extra))
