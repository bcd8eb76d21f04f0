"""Seeded synthetic inputs for single-precision GEMM, C = op(A) * op(B).

This module only draws numbers and lays them out in memory.  It holds none of
the GEMM arithmetic, so both the CPU oracle tests and the CUDA path can consume
exactly the same bits.

Storage convention (row-major throughout, as in the GEMM definition of
"CUDA GEMM operator performance optimization", section 1.1, and the matrix
multiply of the DD2360 workbook, section 9.4):

* A with transA == 0 is stored M x K, element (i, k) at A[i*lda + k], lda >= K.
* A with transA == 1 is stored K x M, element (i, k) at A[k*lda + i], lda >= M.
* B with transB == 0 is stored K x N, element (k, j) at B[k*ldb + j], ldb >= N.
* B with transB == 1 is stored N x K, element (k, j) at B[j*ldb + k], ldb >= K.
* C is stored M x N, element (i, j) at C[i*ldc + j], ldc >= N.

Every buffer is returned as a 2-D (or 3-D for batches) float32 array whose last
axis is the leading dimension, so padding columns exist physically.  Padding
is filled with NaN when ``poison`` is set so that any read of it shows up in
the result.

Random streams: NumPy PCG64 seeded by ``SeedSequence(seed, spawn_key=(key,))``;
A is drawn first, then B, both in their logical (op) order so the values do
not depend on the storage layout.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get", "make_operands", "make_case",
           "flops", "min_bytes"]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One GEMM problem shape, layout and value distribution."""
    name: str
    M: int
    N: int
    K: int
    batch: int = 1
    transA: int = 0
    transB: int = 0
    lda: Optional[int] = None
    ldb: Optional[int] = None
    ldc: Optional[int] = None
    dist: str = "uniform"          # "uniform" U[-1,1), "int" {-4..4}, "normal" N(0, sigma^2)
    sigma: float = 1.0
    poison: bool = False           # NaN in every padding element of A, B and C
    key: int = 0                   # stream key of the PCG64 SeedSequence

    def lds(self):
        lda = self.lda if self.lda is not None else (self.M if self.transA else self.K)
        ldb = self.ldb if self.ldb is not None else (self.K if self.transB else self.N)
        ldc = self.ldc if self.ldc is not None else self.N
        return lda, ldb, ldc

    @property
    def gflop(self) -> float:
        return flops(self.M, self.N, self.K, self.batch) / 1e9


def flops(M: int, N: int, K: int, batch: int = 1) -> int:
    """2*M*N*K per product: K multiplies and K adds per output element
    ("CUDA GEMM operator performance optimization", section 1.1)."""
    return 2 * M * N * K * batch


def min_bytes(M: int, N: int, K: int, batch: int = 1, elem: int = 4) -> int:
    """Compulsory traffic: read A and B once, write C once."""
    return elem * (M * K + K * N + M * N) * batch


def _w(*args, **kw) -> Workload:
    return Workload(*args, **kw)


# The workloads the pages' measurements use, restated as synthetic problems.
# The stream key is the position in this list; nothing else depends on it.
WORKLOADS = {w.name: w for w in [
    _w("sgemm_256x256x256_uniform", 256, 256, 256, dist="uniform", key=0),
    _w("sgemm_256x256x256_int", 256, 256, 256, dist="int", key=1),
    _w("sgemm_3072x3072x3072_uniform", 3072, 3072, 3072, dist="uniform", key=2),
    _w("sgemm_3072x3072x3072_int", 3072, 3072, 3072, dist="int", key=3),
    _w("sgemm_8192x8192x4096_uniform", 8192, 8192, 4096, dist="uniform", key=4),
    _w("sgemm_4096x4096x8192_uniform", 4096, 4096, 8192, dist="uniform", key=5),
    _w("sgemm_8192x8192x8192_uniform", 8192, 8192, 8192, dist="uniform", key=6),
    _w("sgemm_2049x3071x1537_tA_normal", 2049, 3071, 1537, transA=1,
       lda=2052, ldb=3072, ldc=3072, dist="normal", poison=True, key=7),
    _w("sgemm_2049x3071x1537_tA_int", 2049, 3071, 1537, transA=1,
       lda=2052, ldb=3072, ldc=3072, dist="int", poison=True, key=8),
    _w("sgemm_batched96_512x512x64_qkT_normal", 512, 512, 64, batch=96,
       transB=1, dist="normal", sigma=0.125, key=9),
]}


def get(name: str) -> Workload:
    return WORKLOADS[name]


def _rng(seed: int, key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=(key,))))


def _draw(rng: np.random.Generator, shape, dist: str, sigma: float) -> np.ndarray:
    if dist == "uniform":
        # float32 in [0,1) on a 2^-24 grid; 2x-1 is exact in float32, so the
        # result lies in [-1, 1) on a 2^-23 grid.
        return rng.random(shape, dtype=np.float32) * np.float32(2) - np.float32(1)
    if dist == "int":
        return rng.integers(-4, 5, size=shape).astype(np.float32)
    if dist == "normal":
        return (rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)).astype(np.float32)
    if dist == "ones":
        return np.ones(shape, dtype=np.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def _store(logical: np.ndarray, trans: int, ld: int, poison: bool) -> np.ndarray:
    """Lay out a logical (batch, R, S) operand; trans stores it as (batch, S, R)."""
    src = np.swapaxes(logical, 1, 2) if trans else logical
    b, rows, cols = src.shape
    if ld < cols:
        raise ValueError(f"leading dimension {ld} < {cols}")
    if not trans and ld == cols:
        return logical          # already in storage order, no padding to fill
    fill = np.nan if poison else 0.0
    out = np.full((b, rows, ld), fill, dtype=np.float32)
    out[:, :, :cols] = src
    return out


def make_operands(M: int, N: int, K: int, *, batch: int = 1, transA: int = 0,
                  transB: int = 0, lda: Optional[int] = None, ldb: Optional[int] = None,
                  ldc: Optional[int] = None, dist: str = "uniform", sigma: float = 1.0,
                  poison: bool = False, seed: int = 0, key: int = 0) -> dict:
    """Draw op(A) (M x K) then op(B) (K x N) for every batch and store them.

    Returns a dict with the stored buffers ``A`` (batch, rows, lda), ``B``
    (batch, rows, ldb), a ``C`` buffer (batch, M, ldc) pre-filled with NaN when
    ``poison`` (zeros otherwise), the leading dimensions and the logical
    operands ``opA`` (batch, M, K) and ``opB`` (batch, K, N).
    """
    wl = Workload("adhoc", M, N, K, batch=batch, transA=transA, transB=transB,
                  lda=lda, ldb=ldb, ldc=ldc, dist=dist, sigma=sigma, poison=poison, key=key)
    lda, ldb, ldc = wl.lds()
    rng = _rng(seed, key)
    opA = _draw(rng, (batch, M, K), dist, sigma)
    opB = _draw(rng, (batch, K, N), dist, sigma)
    A = _store(opA, transA, lda, poison)
    B = _store(opB, transB, ldb, poison)
    C = np.full((batch, M, ldc), np.nan if poison else 0.0, dtype=np.float32)
    return dict(A=A, B=B, C=C, opA=opA, opB=opB, M=M, N=N, K=K, batch=batch,
                transA=transA, transB=transB, lda=lda, ldb=ldb, ldc=ldc)


def make_case(w: Workload | str, seed: int = 0) -> dict:
    """Operands for a named workload (see WORKLOADS)."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    lda, ldb, ldc = w.lds()
    return make_operands(w.M, w.N, w.K, batch=w.batch, transA=w.transA, transB=w.transB,
                         lda=lda, ldb=ldb, ldc=ldc, dist=w.dist, sigma=w.sigma,
                         poison=w.poison, seed=seed, key=w.key)
