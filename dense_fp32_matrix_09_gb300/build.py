"""Builds libsgemm.so (the CUDA library behind include/sgemm.h) in-tree.

Each translation unit under csrc/ is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``), in parallel, then linked into
``_build/libsgemm.so`` next to this file.  A rebuild happens only when a
source or header is newer than the library.  Next to it, the host compiler
builds ``_build/_sgemm_calls.so`` from csrc/pycalls.c: the CPython module that
marshals the arguments of the binding's two enqueue calls (the binding falls
back to ctypes without it).
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libsgemm.so")
# The same sources with the device-side index checks compiled in
# (-DSGEMM_DEVICE_CHECKS): a separate build, used by its own tests.
BUILD_CHECKED = os.path.join(HERE, "_build_checks")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libsgemm_checks.so")
CHECK_FLAGS = ["-DSGEMM_DEVICE_CHECKS"]
# The CPython argument-marshalling module for sgemm_run / sgemm_run_ex
CALLS_SRC = os.path.join(CSRC, "pycalls.c")
CALLS = os.path.join(BUILD, "_sgemm_calls.so")
calls_build_error: str | None = None

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-Wall,-Wextra", "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the SGEMM library cannot be built")


def build_calls(force: bool = False) -> str | None:
    """Compile the argument-marshalling module with the host compiler (no
    CUDA, no torch); returns its path, or None (with the reason in
    calls_build_error) when it cannot be built here."""
    global calls_build_error
    if not force and os.path.exists(CALLS) and os.path.getmtime(CALLS) >= os.path.getmtime(CALLS_SRC):
        return CALLS
    import sysconfig
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    include = sysconfig.get_paths().get("include", "")
    if not cc or not os.path.exists(os.path.join(include, "Python.h")):
        calls_build_error = "no host compiler or no Python.h"
        return None
    os.makedirs(BUILD, exist_ok=True)
    tmp = CALLS + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-O2", "-shared", "-fPIC", "-Wall", "-I" + include, CALLS_SRC, "-o", tmp, "-ldl"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        calls_build_error = (r.stdout + r.stderr)[-2000:]
        return None
    os.replace(tmp, CALLS)
    calls_build_error = None
    return CALLS


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile and link the library (checked: the build with the device-side
    index checks, in its own directory); returns its path."""
    out_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    build_calls(force)
    if not force and not is_stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    flags = NVCC_FLAGS + GENCODE + (CHECK_FLAGS if checked else []) + list(extra_flags or [])
    objs = []

    def compile_one(src: str) -> str:
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [cc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([cc, "-shared", *GENCODE, "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
