"""Build libdiffattn.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit under csrc/ is compiled in parallel to an object
file, then the objects are linked into ``libdiffattn.so`` next to this file.
Objects live in ``_build/`` (git-ignored).  Set ``DIFFATTN_PTXAS_VERBOSE=1``
to print register / spill / shared-memory usage per kernel.

``build(debug=True)`` makes ``libdiffattn_debug.so`` from the same sources
with ``-DDA_DEBUG_CHECKS`` (objects in ``_build/debug/``): the kernels test
the indices they write through and record failures in the error word.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libdiffattn.so")
LIB_DEBUG = os.path.join(HERE, "libdiffattn_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libdiffattn.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    out = [os.path.join(INCLUDE, "diffattn.h")]
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return out


def _compile(src: str, verbose: bool, debug: bool = False) -> str:
    obj = os.path.join(BUILD, "debug" if debug else "", os.path.basename(src)[:-3] + ".o")
    newest_dep = max(os.path.getmtime(p) for p in _deps() + [src])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest_dep:
        return obj
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj + ".tmp"]
    if debug:
        cmd.append("-DDA_DEBUG_CHECKS")
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose: bool | None = None, debug: bool = False) -> str:
    """Compile every kernel for sm_103a and link libdiffattn.so (or, with
    debug=True, libdiffattn_debug.so); returns its path."""
    if verbose is None:
        verbose = os.environ.get("DIFFATTN_PTXAS_VERBOSE") == "1"
    objdir = os.path.join(BUILD, "debug") if debug else BUILD
    lib = LIB_DEBUG if debug else LIB
    os.makedirs(objdir, exist_ok=True)
    if force:
        for f in os.listdir(objdir):
            if f.endswith(".o"):
                os.remove(os.path.join(objdir, f))
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug), srcs))
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs)):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))
