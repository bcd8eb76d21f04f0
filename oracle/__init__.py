"""CPU oracle for single-precision GEMM -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it;
the two share no code.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, fp64 accumulation in
ascending k, one rounding to fp32 at the end), which follows the GEMM
definition in "CUDA GEMM operator performance optimization", section 1.1, and
the double-accumulating CPU reference of the DD2360 workbook, section 14.3
lab.  This module builds it with gcc, loads it with ctypes and wraps it for
NumPy arrays laid out as described in ``workloads``.

Every function here is pinned by the CPU tests in ``tests/test_oracle_pins.py``
(closed forms, exact integer products, exact rational brute force, a library
routine, layout invariants and planted-mistake checks).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "sgemm_oracle.c")
LIB = os.path.join(_HERE, "liboracle_sgemm.so")

_i64 = ctypes.c_int64
_int = ctypes.c_int
_fp = ctypes.POINTER(ctypes.c_float)
_dp = ctypes.POINTER(ctypes.c_double)
_lp = ctypes.POINTER(ctypes.c_int64)

_lib = None


def compile_oracle(src: str = SRC, out: str = LIB) -> str:
    """Compile the C oracle into a shared library (strict IEEE: no fast-math)."""
    cmd = ["gcc", "-O3", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-pthread", src, "-o", out + ".tmp", "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(out + ".tmp", out)
    return out


def load(path: str = LIB, *, rebuild: bool = False):
    """Load (building first if needed) an oracle library and declare its ABI."""
    global _lib
    if path == LIB and _lib is not None and not rebuild:
        return _lib
    if rebuild or not os.path.exists(path) or (
            path == LIB and os.path.getmtime(path) < os.path.getmtime(SRC)):
        compile_oracle(SRC if path == LIB else path[:-3] + ".c", path)
    lib = ctypes.CDLL(path)
    lib.oracle_sgemm.restype = _int
    lib.oracle_sgemm.argtypes = [_i64, _i64, _i64, _fp, _i64, _int, _fp, _i64, _int,
                                 _fp, _i64, _dp, _i64, _int]
    lib.oracle_sgemm_strided_batched.restype = _int
    lib.oracle_sgemm_strided_batched.argtypes = [
        _i64, _i64, _i64, _fp, _i64, _i64, _int, _fp, _i64, _i64, _int,
        _fp, _i64, _i64, _dp, _i64, _i64, _i64, _int]
    lib.oracle_sgemm_entries.restype = _int
    lib.oracle_sgemm_entries.argtypes = [_i64, _i64, _i64, _fp, _i64, _int, _fp, _i64, _int,
                                         _i64, _lp, _lp, _fp, _dp]
    lib.oracle_sgemm_ex.restype = _int
    lib.oracle_sgemm_ex.argtypes = [_i64, _i64, _i64, ctypes.c_double, _fp, _i64, _int, _fp, _i64,
                                    _int, ctypes.c_double, _fp, _i64, _fp, _fp, _i64, _dp, _i64]
    if path == LIB:
        _lib = lib
    return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _f32(a: np.ndarray) -> np.ndarray:
    if a.dtype != np.float32 or not a.flags.c_contiguous:
        raise TypeError("oracle buffers must be C-contiguous float32")
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctype)


def sgemm(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, *, transA: int = 0,
          transB: int = 0, lda: Optional[int] = None, ldb: Optional[int] = None,
          with_scale: bool = False, nthreads: Optional[int] = None, lib=None):
    """C = op(A) op(B) for one problem, stored buffers in, dense M x N out.

    ``A``/``B`` are the stored buffers (any shape; their memory is read with
    the given leading dimensions).  Returns C (float32, M x N) and, when
    ``with_scale``, S = sum_k |a||b| (float64, M x N).
    """
    lib = lib or load()
    A = _f32(np.ascontiguousarray(A))
    B = _f32(np.ascontiguousarray(B))
    lda = lda if lda is not None else (M if transA else K)
    ldb = ldb if ldb is not None else (K if transB else N)
    C = np.zeros((M, N), dtype=np.float32)
    S = np.zeros((M, N), dtype=np.float64) if with_scale else None
    st = lib.oracle_sgemm(M, N, K, _ptr(A, _fp), lda, transA, _ptr(B, _fp), ldb, transB,
                          _ptr(C, _fp), N, _ptr(S, _dp) if S is not None else None, N,
                          nthreads or default_threads())
    if st:
        raise RuntimeError(f"oracle_sgemm failed with status {st}")
    return (C, S) if with_scale else C


def sgemm_strided_batched(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, batch: int, *,
                          transA: int = 0, transB: int = 0, lda: Optional[int] = None,
                          ldb: Optional[int] = None, strideA: Optional[int] = None,
                          strideB: Optional[int] = None, with_scale: bool = False,
                          nthreads: Optional[int] = None, lib=None):
    """Batched product; returns C (batch, M, N) [and S (batch, M, N)]."""
    lib = lib or load()
    A = _f32(np.ascontiguousarray(A))
    B = _f32(np.ascontiguousarray(B))
    lda = lda if lda is not None else (M if transA else K)
    ldb = ldb if ldb is not None else (K if transB else N)
    strideA = strideA if strideA is not None else (A.size // max(batch, 1))
    strideB = strideB if strideB is not None else (B.size // max(batch, 1))
    C = np.zeros((batch, M, N), dtype=np.float32)
    S = np.zeros((batch, M, N), dtype=np.float64) if with_scale else None
    st = lib.oracle_sgemm_strided_batched(
        M, N, K, _ptr(A, _fp), lda, strideA, transA, _ptr(B, _fp), ldb, strideB, transB,
        _ptr(C, _fp), N, M * N, _ptr(S, _dp) if S is not None else None, N, M * N,
        batch, nthreads or default_threads())
    if st:
        raise RuntimeError(f"oracle_sgemm_strided_batched failed with status {st}")
    return (C, S) if with_scale else C


def sgemm_entries(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, rows, cols, *,
                  transA: int = 0, transB: int = 0, lda: Optional[int] = None,
                  ldb: Optional[int] = None, lib=None):
    """C(rows[t], cols[t]) and S(rows[t], cols[t]) one dot product at a time."""
    lib = lib or load()
    A = _f32(np.ascontiguousarray(A))
    B = _f32(np.ascontiguousarray(B))
    lda = lda if lda is not None else (M if transA else K)
    ldb = ldb if ldb is not None else (K if transB else N)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if rows.shape != cols.shape:
        raise ValueError("rows and cols differ in shape")
    out = np.zeros(rows.shape, dtype=np.float32)
    sab = np.zeros(rows.shape, dtype=np.float64)
    st = lib.oracle_sgemm_entries(M, N, K, _ptr(A, _fp), lda, transA, _ptr(B, _fp), ldb, transB,
                                  rows.size, _ptr(rows, _lp), _ptr(cols, _lp),
                                  _ptr(out, _fp), _ptr(sab, _dp))
    if st:
        raise RuntimeError(f"oracle_sgemm_entries failed with status {st}")
    return out, sab


def sgemm_ex(A: np.ndarray, B: np.ndarray, M: int, N: int, K: int, *, alpha: float = 1.0,
             beta: float = 0.0, C_in: Optional[np.ndarray] = None, bias: Optional[np.ndarray] = None,
             transA: int = 0, transB: int = 0, lda: Optional[int] = None,
             ldb: Optional[int] = None, lib=None):
    """C = alpha op(A) op(B) + beta C_in + bias (bias per column), formed in fp64
    and rounded once; returns (C, S) with the tolerance scale S.  One dot
    product per output (single thread): for small and medium problems."""
    lib = lib or load()
    A = _f32(np.ascontiguousarray(A))
    B = _f32(np.ascontiguousarray(B))
    lda = lda if lda is not None else (M if transA else K)
    ldb = ldb if ldb is not None else (K if transB else N)
    if beta != 0.0:
        C_in = _f32(np.ascontiguousarray(C_in))
        ldc_in = C_in.shape[-1]
    else:
        ldc_in = N
    if bias is not None:
        bias = _f32(np.ascontiguousarray(bias))
    C = np.zeros((M, N), dtype=np.float32)
    S = np.zeros((M, N), dtype=np.float64)
    st = lib.oracle_sgemm_ex(M, N, K, alpha, _ptr(A, _fp), lda, transA, _ptr(B, _fp), ldb, transB,
                             beta, _ptr(C_in, _fp) if beta != 0.0 else None, ldc_in,
                             _ptr(bias, _fp) if bias is not None else None,
                             _ptr(C, _fp), N, _ptr(S, _dp), N)
    if st:
        raise RuntimeError(f"oracle_sgemm_ex failed with status {st}")
    return C, S


# Acceptance bound for fp32 results against the oracle, elementwise:
# |C - C_ref| <= REL_TOL * sum_k |a_ik||b_kj| + ABS_TOL.
REL_TOL = 1e-5
ABS_TOL = 1e-6


def within_tolerance(C: np.ndarray, C_ref: np.ndarray, S: np.ndarray,
                     rel: float = REL_TOL, abs_: float = ABS_TOL) -> np.ndarray:
    """Boolean mask of outputs inside the bound (NaN anywhere fails)."""
    diff = np.abs(C.astype(np.float64) - C_ref.astype(np.float64))
    return diff <= rel * S + abs_


def rrmse(C: np.ndarray, C_ref: np.ndarray) -> float:
    """sqrt(sum (C - C_ref)^2 / sum C_ref^2): the relative RMS error that the
    ChetanC28/cuda-kernels page reports for its FMA and TF32 kernels."""
    d = C.astype(np.float64) - C_ref.astype(np.float64)
    den = float(np.sum(C_ref.astype(np.float64) ** 2))
    return float(np.sqrt(np.sum(d * d) / den)) if den > 0 else float(np.sqrt(np.sum(d * d)))
