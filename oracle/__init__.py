"""CPU oracle for C = A x B (row-major FP32, fp64 accumulation).

TEST INFRASTRUCTURE ONLY: ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` may import this module; the CUDA library and its Python
binding never do.  The arithmetic lives in ``tg_oracle.c`` (see its header for
the definition and the readings of the pages); this file only compiles it with
gcc and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tg_oracle.c")
_LIB = os.path.join(_HERE, "libtg_oracle.so")

# -ffp-contract=off: the oracle's additions are plain double adds.  (A fused
# multiply-add would give the same result anyway because a float x float
# product is exact in double, but the flag keeps the source's meaning literal.)
CFLAGS = ["-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off"]

_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc."""
    cmd = ["gcc", *CFLAGS, *extra_flags, src, "-o", out]
    subprocess.run(cmd, check=True)
    return out


def _needs_build() -> bool:
    return (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def load(path: str | None = None):
    """Load (building first if stale) and return the ctypes library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        if _needs_build():
            build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def _declare(lib):
    i64, fp = ctypes.c_int64, ctypes.c_void_p
    lib.tg_oracle_sgemm.argtypes = [i64, i64, i64, fp, i64, fp, i64, fp, i64]
    lib.tg_oracle_sgemm.restype = ctypes.c_int
    lib.tg_oracle_sgemm_rows.argtypes = [i64, fp, i64, i64, i64, fp, i64, fp, i64, fp, i64]
    lib.tg_oracle_sgemm_rows.restype = ctypes.c_int
    lib.tg_oracle_sgemm_general.argtypes = [ctypes.c_int, ctypes.c_int, i64, i64, i64, ctypes.c_float, fp, i64,
                                            fp, i64, ctypes.c_float, fp, i64]
    lib.tg_oracle_sgemm_general.restype = ctypes.c_int
    lib.tg_oracle_transpose.argtypes = [i64, i64, fp, i64, fp, i64]
    lib.tg_oracle_transpose.restype = ctypes.c_int
    lib.tg_oracle_sum.argtypes = [i64, fp, fp]
    lib.tg_oracle_sum.restype = ctypes.c_int
    lib.tg_oracle_threads.argtypes = []
    lib.tg_oracle_threads.restype = ctypes.c_int
    lib.tg_oracle_set_threads.argtypes = [ctypes.c_int]
    lib.tg_oracle_set_threads.restype = ctypes.c_int
    return lib


def _as_rowmajor_f32(x: np.ndarray, name: str) -> tuple[np.ndarray, int]:
    if x.dtype != np.float32 or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if x.shape[1] > 1 and x.strides[1] != 4:
        x = np.ascontiguousarray(x)
    ld = x.strides[0] // 4 if x.shape[0] > 1 else max(x.shape[1], 1)
    return x, max(ld, x.shape[1], 1)


def sgemm(A: np.ndarray, B: np.ndarray, out: np.ndarray | None = None, lib=None) -> np.ndarray:
    """C = A @ B for 2-D float32 arrays (row strides may exceed the width)."""
    lib = lib or load()
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    if out is None:
        out = np.empty((M, N), dtype=np.float32)
    C, ldc = _as_rowmajor_f32(out, "out")
    if C.shape != (M, N) or C is not out:
        raise ValueError("out must be an (M, N) float32 array with unit column stride")
    rc = lib.tg_oracle_sgemm(M, N, K, A.ctypes.data, lda, B.ctypes.data, ldb, C.ctypes.data, ldc)
    if rc != 0:
        raise RuntimeError(f"tg_oracle_sgemm failed with code {rc}")
    return out


def sgemm_rows(A: np.ndarray, B: np.ndarray, rows, lib=None) -> np.ndarray:
    """Rows ``rows`` of A @ B, as a (len(rows), N) float32 array."""
    lib = lib or load()
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError(f"inner dimensions differ: {A.shape} x {B.shape}")
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.shape[0], N), dtype=np.float32)
    rc = lib.tg_oracle_sgemm_rows(rows.shape[0], rows.ctypes.data, M, N, K, A.ctypes.data, lda,
                                  B.ctypes.data, ldb, out.ctypes.data, max(N, 1))
    if rc != 0:
        raise RuntimeError(f"tg_oracle_sgemm_rows failed with code {rc}")
    return out


def sgemm_general(op_a: int, op_b: int, alpha: float, A: np.ndarray, B: np.ndarray, beta: float,
                  C: np.ndarray, lib=None) -> np.ndarray:
    """C = alpha * op(A) @ op(B) + beta * C in place (op = transpose when the
    flag is 1); A and B are the stored matrices.  Returns C."""
    lib = lib or load()
    A, lda = _as_rowmajor_f32(A, "A")
    B, ldb = _as_rowmajor_f32(B, "B")
    M, K = (A.shape[1], A.shape[0]) if op_a else A.shape
    Kb, N = (B.shape[1], B.shape[0]) if op_b else B.shape
    if Kb != K:
        raise ValueError("inner dimensions differ")
    Cv, ldc = _as_rowmajor_f32(C, "C")
    if Cv is not C or C.shape != (M, N):
        raise ValueError("C must be an (M, N) float32 array with unit column stride")
    rc = lib.tg_oracle_sgemm_general(int(op_a), int(op_b), M, N, K, float(alpha), A.ctypes.data, lda,
                                     B.ctypes.data, ldb, float(beta), C.ctypes.data, ldc)
    if rc != 0:
        raise RuntimeError(f"tg_oracle_sgemm_general failed with code {rc}")
    return C


def transpose(X: np.ndarray, lib=None) -> np.ndarray:
    """X^T (cols x rows, contiguous) by the oracle's index permutation."""
    lib = lib or load()
    X, ld = _as_rowmajor_f32(X, "X")
    rows, cols = X.shape
    out = np.empty((cols, rows), dtype=np.float32)
    rc = lib.tg_oracle_transpose(rows, cols, X.ctypes.data, ld, out.ctypes.data, max(rows, 1))
    if rc != 0:
        raise RuntimeError(f"tg_oracle_transpose failed with code {rc}")
    return out


def reduce_sum(x: np.ndarray, lib=None) -> np.float32:
    """Sum of a 1-D float32 array (double accumulation, one rounding)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    out = np.zeros(1, dtype=np.float32)
    rc = lib.tg_oracle_sum(x.shape[0], x.ctypes.data, out.ctypes.data)
    if rc != 0:
        raise RuntimeError(f"tg_oracle_sum failed with code {rc}")
    return out[0]


def threads(lib=None) -> int:
    """OpenMP threads the oracle uses."""
    return int((lib or load()).tg_oracle_threads())


def set_threads(n: int, lib=None) -> int:
    """Use n OpenMP threads in later calls (timing only); returns the count."""
    return int((lib or load()).tg_oracle_set_threads(int(n)))
