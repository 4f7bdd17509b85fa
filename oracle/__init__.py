"""Oracle for C = alpha*A*B + beta*C (FP64 accumulation, CPU, plain C).

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference leg of ``bench.py``; never by the library
package.  It shares no code with the CUDA path: the arithmetic lives in
``sgemm_ref.c`` and this module only compiles it and passes numpy buffers.

The definition followed is the one on the page "Deep dive into the sgemmNN
algorithm" (lazypool blog), section "Why SGEMM matters": A is m x k, B is
k x n, C is m x n, C = alpha * A x B + beta * C; storage is row-major with
leading dimensions (row-major indexing of the naive kernel on page
m.lqnn.cn/news/94381, section 1.1).  See ``sgemm_ref.c`` for the rounding
rules and the BLAS conventions for alpha == 0 and beta == 0.

Pins: every function here is checked in ``tests/test_oracle.py`` against
closed forms (identity, all-ones), invariants (alpha = 0, beta = 0,
transposition), exact integer arithmetic, a hand-expanded 2 x 2 case and
numpy's float64 matmul on tiny shapes; ``tests/test_oracle_mutants.py``
plants plausible mistakes in a copy of the C source and checks that the pins
catch each one.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "sgemm_ref.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

CFLAGS = ["-O3", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_lib = None


def compile_oracle(source: str = SOURCE, out: str = LIB_PATH) -> str:
    """Compile ``source`` (default: the oracle) into a shared library at ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    i64 = ctypes.c_int64
    fp = ctypes.c_void_p
    lib.oracle_sgemm.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                 fp, i64, fp, i64, ctypes.c_float, fp, i64]
    lib.oracle_sgemm.restype = ctypes.c_int
    lib.oracle_sgemm_f64.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                     fp, i64, fp, i64, ctypes.c_float, fp, i64, fp, i64]
    lib.oracle_sgemm_f64.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
    lib.oracle_set_num_threads.restype = None
    return lib


def load_library(path: str) -> ctypes.CDLL:
    """Load a compiled oracle (or a planted-mistake copy of it) from ``path``."""
    return _declare(ctypes.CDLL(path))


def lib() -> ctypes.CDLL:
    """The oracle library, compiled on first use if it is missing or stale."""
    global _lib
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(LIB_PATH)
                     or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE))
            if stale:
                compile_oracle()
            _lib = load_library(LIB_PATH)
        return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle buffers must be contiguous"
    return a.ctypes.data


def _check_extent(buf, rows, cols, ld, name):
    if rows > 0 and cols > 0:
        need = (rows - 1) * ld + cols
        if buf is None or buf.size < need:
            raise ValueError(f"{name}: buffer of {0 if buf is None else buf.size} elements "
                             f"is smaller than ({rows}-1)*{ld}+{cols}={need}")


def sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, *, library=None):
    """C <- (float)(alpha*A*B + beta*C) in place on flat float32 numpy buffers.

    ``A``, ``B``, ``C`` are C-contiguous float32 arrays (any shape) holding the
    row-major matrices at leading dimensions ``lda``, ``ldb``, ``ldc``.
    """
    lib_ = library or lib()
    for x in (A, B):
        assert x is None or x.dtype == np.float32
    assert C.dtype == np.float32
    if alpha != 0 and K > 0:
        _check_extent(A, M, K, lda, "A")
        _check_extent(B, K, N, ldb, "B")
    _check_extent(C, M, N, ldc, "C")
    rc = lib_.oracle_sgemm(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc)
    if rc != 0:
        raise ValueError(f"oracle_sgemm rejected its arguments (status {rc})")
    return C


def sgemm_f64(M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc0, *, library=None):
    """Unrounded result D = alpha*A*B + beta*C0 as a dense (M, N) float64 array."""
    lib_ = library or lib()
    D = np.empty((M, N), dtype=np.float64)
    if alpha != 0 and K > 0:
        _check_extent(A, M, K, lda, "A")
        _check_extent(B, K, N, ldb, "B")
    if beta != 0:
        _check_extent(C0, M, N, ldc0, "C0")
    rc = lib_.oracle_sgemm_f64(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta,
                               _ptr(C0), ldc0, _ptr(D), max(N, 1))
    if rc != 0:
        raise ValueError(f"oracle_sgemm_f64 rejected its arguments (status {rc})")
    return D


def sgemm_rows(rows, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, *, library=None):
    """Float results of the output rows ``rows`` only, as a (len(rows), N) array.

    The listed rows of A (and of C0) are gathered into a contiguous
    len(rows) x K matrix and passed to the oracle in one call; each output
    row is computed exactly as a full ``sgemm`` call would compute it (rows
    are independent).  This is how outputs of shapes too large for the full
    oracle are sampled.
    """
    rows = [int(i) for i in rows]
    R = len(rows)
    reads_ab = alpha != 0 and K > 0
    a = np.empty((R, max(K, 1)), dtype=np.float32)
    if reads_ab:
        for r, i in enumerate(rows):
            a[r, :K] = A[i * lda:i * lda + K]
    c = np.full((R, max(N, 1)), np.nan, dtype=np.float32)
    if beta != 0:
        for r, i in enumerate(rows):
            c[r, :N] = C0[i * ldc:i * ldc + N]
    sgemm(R, N, K, alpha, a.reshape(-1) if reads_ab else None, max(K, 1), B, ldb, beta,
          c.reshape(-1), max(N, 1), library=library)
    return c[:, :N]


def num_threads(library=None) -> int:
    return (library or lib()).oracle_num_threads()


def set_num_threads(n: int, library=None) -> None:
    (library or lib()).oracle_set_num_threads(n)
