"""CPU oracle for C = A·B (+bias): test infrastructure only.

Only the test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA library
and never imports it.

``gemm``/``gemm_rows`` wrap ``gemm_oracle.c`` (plain triple loop, binary64
accumulation, ascending k).  ``schedule`` holds the plain readings of the two
scheduling rules the pages give (Stream-K range split, ``storage_align``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compiles the C oracle with gcc (no fast-math, no FMA contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    os.makedirs(_LIB_DIR, exist_ok=True)
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_gemm_rows.restype = ctypes.c_int
        lib.oracle_gemm_rows.argtypes = [
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def f16_to_f64(code: int) -> float:
    """Decodes one binary16 bit pattern (0..65535) to binary64."""
    return _load().oracle_f16_to_f64(int(code))


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float16:
        return 0
    if a.dtype == np.float32:
        return 1
    raise TypeError("oracle inputs are float16 or float32, got %s" % a.dtype)


def _dims(A, B, a_major, b_major):
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("A and B are 2-D storage arrays")
    M, K = A.shape if a_major == 0 else A.shape[::-1]
    Kb, N = B.shape if b_major == 0 else B.shape[::-1]
    if K != Kb:
        raise ValueError("inner dimensions differ: %d vs %d" % (K, Kb))
    return int(M), int(N), int(K)


def gemm_rows(A: np.ndarray, B: np.ndarray, bias=None, *, a_major: int = 0,
              b_major: int = 0, rows=None, threads: int | None = None) -> np.ndarray:
    """Rows of C = A·B (+bias) in binary64.

    A, B are storage arrays: A has shape (M, K) when ``a_major == 0`` (row-major)
    and (K, M) when ``a_major == 1`` (column-major, i.e. Aᵀ stored row-major);
    B has shape (K, N) when ``b_major == 0`` and (N, K) when ``b_major == 1``.
    ``rows``: None for all rows, else a sequence of row indices.
    Returns an array of shape (len(rows) or M, N), dtype float64.
    """
    A = np.ascontiguousarray(A)
    B = np.ascontiguousarray(B)
    M, N, K = _dims(A, B, a_major, b_major)
    if bias is not None:
        bias = np.ascontiguousarray(bias, dtype=np.float32)
        if bias.shape != (N,):
            raise ValueError("bias has shape %s, expected (%d,)" % (bias.shape, N))
    if rows is None:
        rows_arr = None
        nrows = M
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        nrows = rows_arr.size
    C = np.empty((nrows, N), dtype=np.float64)
    if threads is None:
        threads = host_threads()
    rc = _load().oracle_gemm_rows(
        M, N, K, A.ctypes.data, _dtype_code(A), a_major,
        B.ctypes.data, _dtype_code(B), b_major,
        None if bias is None else bias.ctypes.data,
        None if rows_arr is None else rows_arr.ctypes.data, nrows,
        C.ctypes.data, int(threads))
    if rc != 0:
        raise ValueError("oracle_gemm_rows failed with code %d" % rc)
    return C


def gemm(A, B, bias=None, *, a_major: int = 0, b_major: int = 0,
         threads: int | None = None) -> np.ndarray:
    """The whole product C (M x N, binary64); see ``gemm_rows``."""
    return gemm_rows(A, B, bias, a_major=a_major, b_major=b_major, rows=None,
                     threads=threads)
