"""CPU oracle for C[M x K] = A[M x N] . B[N x K] (float32 in, float64 out).

TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers allowed; the GPU library never imports, links
or runs anything here, and nothing here imports the GPU library.

The arithmetic lives in ``sgemm_oracle.c`` (a plain double-accumulating triple loop,
see its header for the pages' definition it follows). This file only compiles that
source with gcc and marshals numpy arrays to it.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compiles ``sgemm_oracle.c`` into ``oracle/_build/liboracle.so`` (plain gcc, no
    fast-math, no FMA contraction) and returns the library path."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-pthread", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64 = ctypes.c_int64
            vp = ctypes.c_void_p
            lib.oracle_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, ctypes.c_int]
            lib.oracle_gemm.restype = ctypes.c_int
            lib.oracle_entries.argtypes = [vp, vp, i64, i64, i64, vp, vp, i64, vp, vp]
            lib.oracle_entries.restype = ctypes.c_int
            _lib = lib
    return _lib


def _as_f32(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("expected a 2-D array")
    return x


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def gemm(A, B, with_scale: bool = True, threads: int | None = None):
    """Returns (C, S): C = A.B summed in double with n ascending, and S = |A|.|B|
    (or None when ``with_scale`` is False), both float64 M x K arrays."""
    A = _as_f32(A)
    B = _as_f32(B)
    M, N = A.shape
    N2, K = B.shape
    if N != N2:
        raise ValueError(f"inner dimensions differ: {A.shape} . {B.shape}")
    C = np.empty((M, K), dtype=np.float64)
    S = np.empty((M, K), dtype=np.float64) if with_scale else None
    rc = _load().oracle_gemm(A.ctypes.data, B.ctypes.data, C.ctypes.data,
                             S.ctypes.data if S is not None else None,
                             M, N, K, threads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_gemm failed")
    return C, S


def entries(A, B, rows, cols):
    """Returns (C_vals, S_vals) at coordinates (rows[i], cols[i]), each entry summed on
    its own in the same order as :func:`gemm`."""
    A = _as_f32(A)
    B = _as_f32(B)
    M, N = A.shape
    N2, K = B.shape
    if N != N2:
        raise ValueError(f"inner dimensions differ: {A.shape} . {B.shape}")
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape or rows.ndim != 1:
        raise ValueError("rows and cols must be 1-D and the same length")
    c = np.empty(rows.shape[0], dtype=np.float64)
    s = np.empty(rows.shape[0], dtype=np.float64)
    rc = _load().oracle_entries(A.ctypes.data, B.ctypes.data, M, N, K, rows.ctypes.data,
                                cols.ctypes.data, rows.shape[0], c.ctypes.data, s.ctypes.data)
    if rc != 0:
        raise RuntimeError("oracle_entries failed (bad shape or index)")
    return c, s
