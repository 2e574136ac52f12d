"""Build libdcn_b300.so in-tree with nvcc for sm_103a (B300).

Each ``csrc/*.cu`` compiles to an object under ``_build/`` (in parallel), and
the objects link into ``libdcn_b300.so`` next to this file.  Rebuilds only
when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdcn_b300.so")
# The range-checked build (-DDCN_DEBUG_BOUNDS): every data-dependent access
# checked, violations reported as DCN_ERR_INTERNAL; for tests, not for speed.
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libdcn_b300_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-Wall",
                "-I", os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [__file__])


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(d) > t for d in _deps())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link the library if it is missing or stale; return its path.
    debug_bounds: the range-checked build, a separate library."""
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug_bounds else (LIB, BUILD)
    if not force and not _stale(lib):
        return lib
    os.makedirs(bdir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose else []) + (["-DDCN_DEBUG_BOUNDS"] if debug_bounds else [])
    procs, objs = [], []
    for src in _sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [NVCC] + FLAGS + extra + ["-c", src, "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if pr.returncode:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib + ".tmp.%d" % os.getpid()
    subprocess.check_call([NVCC] + ARCH + ["-shared", "-o", tmp] + objs)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))
