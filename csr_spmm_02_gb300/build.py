"""Compile the CUDA library for sm_103a (nvcc only; no CMake, no torch extension).

Each ``csrc/*.cu`` is compiled in its own nvcc process (in parallel), then
linked into ``_lib/libcsr_spmm_gb300.so`` with a static CUDA runtime.  The
library depends on nothing but the CUDA driver at run time.

Two checking builds of the same sources sit beside it (built on demand by
the tests, never loaded by the product path):

* ``bounds``: every B-row gather and every output store checks its address
  against the launch's buffers, skips an access outside them and reports
  SPMM_ERR_OUT_OF_BOUNDS through the error word (``-DSPMM_DEBUG_BOUNDS``);
* ``stage_timeout``: a kernel's first wait for its staged copies gives up
  after one poll, so that the timeout reporting can be tested without a
  hang or a fault (the kernel still waits for the copies before it leaves).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "_lib")
LIBNAME = "libcsr_spmm_gb300.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]
FLAVORS = {"bounds": ["-DSPMM_DEBUG_BOUNDS"], "stage_timeout": ["-DSPMM_STAGE_SPIN_LIMIT=1"]}


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def lib_path(flavor: str | None = None) -> str:
    name = LIBNAME if flavor is None else LIBNAME.replace(".so", f"_{flavor}.so")
    return os.path.join(LIBDIR, name)


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(ROOT, "include", "spmm.h"), os.path.abspath(__file__)]


def up_to_date(flavor: str | None = None) -> bool:
    lib = lib_path(flavor)
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), flavor: str | None = None) -> str:
    """Build the shared library (or one of the checking builds, FLAVORS) if
    any source is newer; return its path."""
    if not force and up_to_date(flavor):
        return lib_path(flavor)
    extra_flags = [*extra_flags, *(FLAVORS[flavor] if flavor else [])]
    objdir = os.path.join(LIBDIR, "obj" if flavor is None else f"obj_{flavor}")
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *CFLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib_path(flavor) + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stderr}")
    os.replace(tmp, lib_path(flavor))
    return lib_path(flavor)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
