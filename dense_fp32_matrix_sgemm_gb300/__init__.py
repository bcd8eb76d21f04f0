"""GB300-native single-precision GEMM: C = op(A) op(B) in float32.

This package is a thin binding over ``libsgemm_gb300.so``, whose C ABI is
declared in ``include/sgemm_gb300.h``.  The binding only marshals arguments:
every step of the product runs in the library's CUDA kernels.  The compute
entry points go through ``_calls``, a small CPython extension bound to the
loaded library's entry points (a fraction of a microsecond per call), when
it was built, else through ctypes (about 0.2 us per argument); the library,
and so every result, is the same either way.  There is no CPU fallback; if
the library has not been built, every call raises ``SgemmUnavailable``.

Low-level names mirror the C ABI (raw device pointers as Python ints, stream
as a ``cudaStream_t`` int or 0).  ``matmul`` is a convenience for torch CUDA
tensors that computes the pointers and leading dimensions and calls
``sgemm_f32`` / ``sgemm_f32_strided_batched``.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = ["SgemmError", "SgemmUnavailable", "load_library", "library_path",
           "sgemm_f32", "sgemm_f32_strided_batched",
           "status_string", "last_error", "version", "matmul", "SGEMM_OK",
           "probe_fp32_fma", "probe_tf32_mma", "probe_out_elems", "sgemm_f32_tf32x3",
           "sgemm_f32_tf32x3_strided_batched", "tf32x3_workspace_size", "device_status",
           "sgemm_f32_tf32x3_noalloc", "tf32x3_noalloc_max_bytes", "sgemm_f32_tf32",
           "sgemm_f32_tf32_strided_batched", "tf32_workspace_size", "sgemm_f32_splitk",
           "splitk_auto_splits", "splitk_workspace_size", "sgemm_f32_ex", "selftest_wait_timeout",
           "sgemm_f32_streamk", "streamk_workspace_size",
           "sgemm_f32_ex_strided_batched", "sgemm_f32_tf32x3_ex", "set_raster_group",
           "set_tf32x3_chunk_k", "marshalling"]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libsgemm_gb300.so")

SGEMM_OK = 0
STATUS_NAMES = {
    0: "SGEMM_OK", 1: "SGEMM_EINVAL_DIM", 2: "SGEMM_EINVAL_LD", 3: "SGEMM_EINVAL_PTR",
    4: "SGEMM_EINVAL_TRANS", 5: "SGEMM_EINVAL_BATCH", 6: "SGEMM_ELAUNCH", 7: "SGEMM_EDEVICE",
    8: "SGEMM_EWORKSPACE",
}

_i64 = ctypes.c_int64
_int = ctypes.c_int
_vp = ctypes.c_void_p

# Exported symbol -> (restype, argtypes).  Kept in step with include/sgemm_gb300.h.
SIGNATURES = {
    "sgemm_f32": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int, _vp]),
    "sgemm_f32_strided_batched": (_int, [_i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
                                         _vp, _i64, _i64, _i64, _int, _int, _vp]),
    "sgemm_status_string": (ctypes.c_char_p, [_int]),
    "sgemm_last_error": (ctypes.c_char_p, []),
    "sgemm_version": (_int, []),
    "sgemm_f32_ex": (_int, [_i64, _i64, _i64, ctypes.c_float, _vp, _i64, _vp, _i64,
                            ctypes.c_float, _vp, _i64, _vp, _int, _int, _vp]),
    "sgemm_f32_ex_strided_batched": (_int, [_i64, _i64, _i64, ctypes.c_float, _vp, _i64, _i64,
                                            _vp, _i64, _i64, ctypes.c_float, _vp, _i64, _i64,
                                            _vp, _i64, _int, _int, _vp]),
    "sgemm_f32_tf32x3_ex": (_int, [_i64, _i64, _i64, ctypes.c_float, _vp, _i64, _vp, _i64,
                                   ctypes.c_float, _vp, _i64, _vp, _int, _int, _vp,
                                   ctypes.c_uint64, _vp]),
    "sgemm_f32_splitk": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int,
                                _int, _vp, ctypes.c_uint64, _vp]),
    "sgemm_f32_splitk_auto_splits": (_int, [_i64, _i64, _i64]),
    "sgemm_f32_streamk": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int,
                                 _vp, ctypes.c_uint64, _vp]),
    "sgemm_f32_streamk_workspace_size": (ctypes.c_uint64, [_i64, _i64, _i64, _int, _int]),
    "sgemm_f32_splitk_workspace_size": (ctypes.c_uint64, [_i64, _i64, _i64, _int]),
    "sgemm_f32_tf32x3": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int,
                                _vp, ctypes.c_uint64, _vp]),
    "sgemm_f32_tf32x3_strided_batched": (_int, [_i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64,
                                                _i64, _vp, _i64, _i64, _i64, _int, _int, _vp,
                                                ctypes.c_uint64, _vp]),
    "sgemm_f32_tf32x3_workspace_size": (ctypes.c_uint64, [_i64, _i64, _i64, _i64]),
    "sgemm_f32_tf32": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int, _int,
                              _vp, ctypes.c_uint64, _vp]),
    "sgemm_f32_tf32_strided_batched": (_int, [_i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64,
                                              _i64, _vp, _i64, _i64, _i64, _int, _int, _vp,
                                              ctypes.c_uint64, _vp]),
    "sgemm_f32_tf32_workspace_size": (ctypes.c_uint64, [_i64, _i64, _i64, _i64]),
    "sgemm_device_status": (_int, [ctypes.POINTER(ctypes.c_uint), _int]),
    "sgemm_f32_tf32x3_noalloc": (_int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _int,
                                        _int, _vp]),
    "sgemm_f32_tf32x3_noalloc_max_bytes": (ctypes.c_uint64, []),
    "sgemm_probe_fp32_fma": (_int, [_int, _i64, _vp, ctypes.POINTER(ctypes.c_double), _vp]),
    "sgemm_probe_out_elems": (_i64, []),
    "sgemm_probe_tf32_mma": (_int, [_i64, _vp, ctypes.POINTER(ctypes.c_double), _vp]),
    "sgemm_selftest_wait_timeout": (_int, [_i64, _vp]),
    "sgemm_set_raster_group": (_int, [_int]),
    "sgemm_set_tf32x3_chunk_k": (_int, [_int]),
}


class SgemmUnavailable(RuntimeError):
    """The CUDA library is missing or cannot be loaded (no fallback exists)."""


class SgemmError(RuntimeError):
    """A call returned a nonzero sgemm_status."""

    def __init__(self, status: int, detail: str):
        self.status = status
        self.detail = detail
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


_lock = threading.Lock()
_lib = None
_api = None   # what the compute wrappers call: the _calls module, else the ctypes library

# Compute entry points that the _calls extension marshals (same names, same
# argument order as the C ABI); everything else goes through ctypes.
FAST_ENTRIES = ("sgemm_f32", "sgemm_f32_strided_batched", "sgemm_f32_ex",
                "sgemm_f32_ex_strided_batched", "sgemm_f32_tf32x3_ex", "sgemm_f32_splitk",
                "sgemm_f32_streamk", "sgemm_f32_tf32x3", "sgemm_f32_tf32x3_strided_batched",
                "sgemm_f32_tf32", "sgemm_f32_tf32_strided_batched", "sgemm_f32_tf32x3_noalloc")


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libsgemm_gb300.so once and declare its symbols."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise SgemmUnavailable(
                f"{_LIB_PATH} is not built; run __graft_entry__.build() or "
                "python -m dense_fp32_matrix_sgemm_gb300._build")
        try:
            lib = ctypes.CDLL(_LIB_PATH)
        except OSError as e:
            raise SgemmUnavailable(f"cannot load {_LIB_PATH}: {e}") from e
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        global _api
        _api = _bind_calls(lib)
        _lib = lib
        return lib


def _bind_calls(lib):
    """The _calls extension bound to this library's entry points, or the
    ctypes library itself when the extension was not built."""
    try:
        from . import _calls
    except ImportError:
        return lib
    _calls.bind({name: ctypes.cast(getattr(lib, name), ctypes.c_void_p).value
                 for name in FAST_ENTRIES})
    return _calls


def marshalling() -> str:
    """'extension' when the compute calls go through the _calls module, else 'ctypes'."""
    load_library()
    return "ctypes" if _api is _lib else "extension"


def _entry():
    """The compute calls' route, loading the library first if needed."""
    if _lib is None:
        load_library()
    return _api


def status_string(status: int) -> str:
    return load_library().sgemm_status_string(status).decode()


def last_error() -> str:
    return load_library().sgemm_last_error().decode()


def version() -> int:
    return load_library().sgemm_version()


def _check(status: int) -> int:
    if status != SGEMM_OK:
        raise SgemmError(status, last_error())
    return status


def sgemm_f32(M, N, K, A, lda, B, ldb, C, ldc, transA=0, transB=0, stream=0, *, check=True):
    """C = op(A) op(B); A, B, C are device pointers (ints).  Returns the status."""
    st = _entry().sgemm_f32(M, N, K, A or 0, lda, B or 0, ldb, C or 0, ldc,
                            transA, transB, stream or 0)
    return _check(st) if check else st


def sgemm_f32_strided_batched(M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                              batch, transA=0, transB=0, stream=0, *, check=True):
    """Strided-batched C_z = op(A_z) op(B_z).  Returns the status."""
    st = _entry().sgemm_f32_strided_batched(
        M, N, K, A or 0, lda, strideA, B or 0, ldb, strideB, C or 0, ldc, strideC,
        batch, transA, transB, stream or 0)
    return _check(st) if check else st


def sgemm_f32_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias=0, transA=0, transB=0,
                 stream=0, *, check=True):
    """C = alpha op(A) op(B) + beta C + bias (bias: device pointer to N floats or 0)."""
    st = _entry().sgemm_f32_ex(M, N, K, alpha, A or 0, lda, B or 0, ldb, beta,
                               C or 0, ldc, bias or 0, transA, transB, stream or 0)
    return _check(st) if check else st


def sgemm_f32_ex_strided_batched(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, beta, C, ldc,
                                 strideC, bias, batch, transA=0, transB=0, stream=0, *,
                                 check=True):
    st = _entry().sgemm_f32_ex_strided_batched(
        M, N, K, alpha, A or 0, lda, strideA, B or 0, ldb, strideB, beta, C or 0, ldc,
        strideC, bias or 0, batch, transA, transB, stream or 0)
    return _check(st) if check else st


def sgemm_f32_tf32x3_ex(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, bias=0, transA=0, transB=0,
                        workspace=0, workspace_bytes=0, stream=0, *, check=True):
    st = _entry().sgemm_f32_tf32x3_ex(M, N, K, alpha, A or 0, lda, B or 0, ldb, beta,
                                      C or 0, ldc, bias or 0, transA, transB,
                                      workspace or 0, workspace_bytes, stream or 0)
    return _check(st) if check else st


def sgemm_f32_streamk(M, N, K, A, lda, B, ldb, C, ldc, transA=0, transB=0, workspace=0,
                      workspace_bytes=0, stream=0, *, check=True):
    """sgemm_f32 with turned operands and the stream-K tile schedule (see include/sgemm_gb300.h)."""
    st = _entry().sgemm_f32_streamk(M, N, K, A or 0, lda, B or 0, ldb, C or 0, ldc,
                                    transA, transB, workspace or 0, workspace_bytes,
                                    stream or 0)
    return _check(st) if check else st


def streamk_workspace_size(M: int, N: int, K: int, transA: int = 0, transB: int = 0) -> int:
    return load_library().sgemm_f32_streamk_workspace_size(M, N, K, transA, transB)


def sgemm_f32_splitk(M, N, K, A, lda, B, ldb, C, ldc, transA=0, transB=0, splits=0, workspace=0,
                     workspace_bytes=0, stream=0, *, check=True):
    """sgemm_f32 with K split into chunks summed in a fixed order (deterministic)."""
    st = _entry().sgemm_f32_splitk(M, N, K, A or 0, lda, B or 0, ldb, C or 0, ldc,
                                   transA, transB, splits, workspace or 0,
                                   workspace_bytes, stream or 0)
    return _check(st) if check else st


def splitk_auto_splits(M, N, K) -> int:
    return load_library().sgemm_f32_splitk_auto_splits(M, N, K)


def splitk_workspace_size(M, N, K, splits=0) -> int:
    return load_library().sgemm_f32_splitk_workspace_size(M, N, K, splits)


def sgemm_f32_tf32x3(M, N, K, A, lda, B, ldb, C, ldc, transA=0, transB=0, workspace=0,
                     workspace_bytes=0, stream=0, *, check=True):
    """C = op(A) op(B) on the tensor cores (3xTF32); ``workspace`` is a device
    pointer of at least tf32x3_workspace_size(M, N, K, 1) bytes."""
    st = _entry().sgemm_f32_tf32x3(M, N, K, A or 0, lda, B or 0, ldb, C or 0,
                                   ldc, transA, transB, workspace or 0, workspace_bytes,
                                   stream or 0)
    return _check(st) if check else st


def sgemm_f32_tf32x3_strided_batched(M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                                     batch, transA=0, transB=0, workspace=0, workspace_bytes=0,
                                     stream=0, *, check=True):
    """Strided-batched 3xTF32 product."""
    st = _entry().sgemm_f32_tf32x3_strided_batched(
        M, N, K, A or 0, lda, strideA, B or 0, ldb, strideB, C or 0, ldc, strideC,
        batch, transA, transB, workspace or 0, workspace_bytes, stream or 0)
    return _check(st) if check else st


def sgemm_f32_tf32x3_noalloc(M, N, K, A, lda, B, ldb, C, ldc, transA=0, transB=0, stream=0, *,
                             check=True):
    """3xTF32 product that allocates nothing: its scratch is the library's
    built-in device array (see include/sgemm_gb300.h for the size limit and
    the rule that overlapping calls race)."""
    st = _entry().sgemm_f32_tf32x3_noalloc(M, N, K, A or 0, lda, B or 0, ldb,
                                           C or 0, ldc, transA, transB, stream or 0)
    return _check(st) if check else st


def tf32x3_noalloc_max_bytes() -> int:
    return load_library().sgemm_f32_tf32x3_noalloc_max_bytes()


def sgemm_f32_tf32(M, N, K, A, lda, B, ldb, C, ldc, transA=0, transB=0, workspace=0,
                   workspace_bytes=0, stream=0, *, check=True):
    """Plain single-TF32 tensor-core product (reduced precision, see the header)."""
    st = _entry().sgemm_f32_tf32(M, N, K, A or 0, lda, B or 0, ldb, C or 0, ldc,
                                 transA, transB, workspace or 0, workspace_bytes,
                                 stream or 0)
    return _check(st) if check else st


def sgemm_f32_tf32_strided_batched(M, N, K, A, lda, strideA, B, ldb, strideB, C, ldc, strideC,
                                   batch, transA=0, transB=0, workspace=0, workspace_bytes=0,
                                   stream=0, *, check=True):
    st = _entry().sgemm_f32_tf32_strided_batched(
        M, N, K, A or 0, lda, strideA, B or 0, ldb, strideB, C or 0, ldc, strideC,
        batch, transA, transB, workspace or 0, workspace_bytes, stream or 0)
    return _check(st) if check else st


def tf32_workspace_size(M, N, K, batch=1) -> int:
    return load_library().sgemm_f32_tf32_workspace_size(M, N, K, batch)


def tf32x3_workspace_size(M, N, K, batch=1) -> int:
    return load_library().sgemm_f32_tf32x3_workspace_size(M, N, K, batch)


def device_status(reset: bool = False) -> int:
    """The library's device status word (bit 0: a tensor-core pipeline wait ran out)."""
    flags = ctypes.c_uint(0)
    _check(load_library().sgemm_device_status(ctypes.byref(flags), 1 if reset else 0))
    return flags.value


def probe_fp32_fma(packed: int, iterations: int, out_ptr: int, stream=0) -> float:
    """Launch the FP32 FMA probe; returns the FLOPs of the launch."""
    flops = ctypes.c_double(0.0)
    _check(load_library().sgemm_probe_fp32_fma(packed, iterations, out_ptr or None,
                                               ctypes.byref(flops), stream or None))
    return flops.value


def probe_tf32_mma(iterations: int, out_ptr: int, stream=0) -> float:
    """Launch the TF32 tensor-pipe probe; returns the FLOPs of the launch."""
    flops = ctypes.c_double(0.0)
    _check(load_library().sgemm_probe_tf32_mma(iterations, out_ptr or None, ctypes.byref(flops),
                                               stream or None))
    return flops.value


def probe_out_elems() -> int:
    return load_library().sgemm_probe_out_elems()


def set_raster_group(group_m: int) -> int:
    """Tile rows per raster group for later calls (0 restores the library's 8);
    returns the previous value (see include/sgemm_gb300_probe.h)."""
    prev = load_library().sgemm_set_raster_group(group_m)
    if prev < 0:
        raise ValueError(f"group_m={group_m}: must be 0 .. 65536")
    return prev


def set_tf32x3_chunk_k(chunk_k: int) -> int:
    """K per chunk of the three-term product over K > 256 for later calls (0
    restores the library's 128); returns the previous value (see
    include/sgemm_gb300_probe.h)."""
    prev = load_library().sgemm_set_tf32x3_chunk_k(chunk_k)
    if prev < 0:
        raise ValueError(f"chunk_k={chunk_k}: must be 0 or a multiple of 32 from 32 to 2^30")
    return prev


def selftest_wait_timeout(limit_cycles: int = 10_000_000, stream=0) -> int:
    """Run the bounded-wait self-test (see include/sgemm_gb300_probe.h)."""
    return _check(load_library().sgemm_selftest_wait_timeout(limit_cycles, stream or None))


def _operand(t, name):
    """Return (rows, cols, ld, trans) for a 2-D/3-D CUDA float32 view: row-major
    storage (unit column stride) is taken as is; a transposed view (unit row
    stride) is passed as the stored matrix with trans = 1."""
    import torch
    if t.dtype != torch.float32 or not t.is_cuda:
        raise TypeError(f"{name} must be a float32 CUDA tensor")
    r, c = t.shape[-2], t.shape[-1]
    sr, sc = t.stride(-2), t.stride(-1)
    if sc == 1 and (sr >= max(1, c) or r <= 1):
        return r, c, max(sr, c, 1), 0
    if sr == 1 and (sc >= max(1, r) or c <= 1):
        return r, c, max(sc, r, 1), 1
    raise ValueError(f"{name} must have one unit stride among its last two dimensions")


def matmul(A, B, out=None, stream=None, precision="fp32", workspace=None, alpha=1.0, beta=0.0,
           bias=None, splits=None):
    """out = alpha * A @ B + beta * out + bias for float32 CUDA tensors of shape
    (M, K) x (K, N), or batched (b, M, K) x (b, K, N); bias has N elements.
    Transposed views are handled through the trans flags without copies.
    Runs on ``stream`` (default: torch's current stream).

    precision="fp32": CUDA-core FMA (sgemm_f32_streamk for single plain
    products, which turns K-contiguous operands of large problems and uses
    stream-K; sgemm_f32_strided_batched for batches; sgemm_f32_ex* with an
    epilogue; sgemm_f32_splitk when ``splits`` is given: 0 = automatic);
    "tf32x3": tensor cores with the three-term TF32 split (sgemm_f32_tf32x3*);
    "tf32": one TF32 product (sgemm_f32_tf32*, reduced precision).  Entries
    that need scratch memory use ``workspace`` (a CUDA uint8 tensor) or a
    fresh one from torch's allocator.  beta != 0 needs ``out`` (its values are
    read)."""
    import torch
    if precision not in ("fp32", "tf32x3", "tf32"):
        raise ValueError("precision must be 'fp32', 'tf32x3' or 'tf32'")
    if A.dim() != B.dim() or A.dim() not in (2, 3):
        raise ValueError("A and B must both be 2-D or both 3-D")
    M, K, lda, tA = _operand(A, "A")
    K2, N, ldb, tB = _operand(B, "B")
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    batched = A.dim() == 3
    batch = A.shape[0] if batched else 1
    if batched and B.shape[0] != batch:
        raise ValueError("batch sizes differ")
    shape = (batch, M, N) if batched else (M, N)
    plain = alpha == 1.0 and beta == 0.0 and bias is None
    if out is None:
        if beta != 0.0:
            raise ValueError("beta != 0 reads out: pass it")
        out = torch.empty(shape, dtype=torch.float32, device=A.device)
    elif tuple(out.shape) != shape or out.dtype != torch.float32 or out.stride(-1) != 1:
        raise ValueError("out has the wrong shape, dtype or layout")
    bp = 0
    if bias is not None:
        if bias.dtype != torch.float32 or not bias.is_cuda or bias.numel() != N or \
                (bias.dim() > 0 and bias.stride(-1) != 1):
            raise ValueError("bias must be a contiguous float32 CUDA tensor of N elements")
        bp = bias.data_ptr()
    ldc = max(out.stride(-2), N, 1)
    s = stream if stream is not None else torch.cuda.current_stream(A.device)
    sp = s.cuda_stream if hasattr(s, "cuda_stream") else int(s)

    def scratch(need):
        nonlocal workspace
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=A.device)
        return workspace.data_ptr(), workspace.numel()

    if splits is not None:
        if precision != "fp32" or batched or not plain:
            raise ValueError("split-K is for single fp32 products without an epilogue")
        ws, wsb = scratch(splitk_workspace_size(M, N, K, splits))
        sgemm_f32_splitk(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, tA,
                         tB, splits, ws, wsb, sp)
    elif precision == "fp32":
        if plain and batched:
            sgemm_f32_strided_batched(M, N, K, A.data_ptr(), lda, A.stride(0), B.data_ptr(), ldb,
                                      B.stride(0), out.data_ptr(), ldc, out.stride(0), batch,
                                      tA, tB, sp)
        elif plain:
            # the fastest CUDA-core path: large problems turn K-contiguous
            # operands and use stream-K, with a workspace; others need none
            need = streamk_workspace_size(M, N, K, tA, tB)
            if need:
                ws, wsb = scratch(need)
                sgemm_f32_streamk(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(),
                                  ldc, tA, tB, ws, wsb, sp)
            else:
                sgemm_f32(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, tA,
                          tB, sp)
        elif batched:
            sgemm_f32_ex_strided_batched(M, N, K, alpha, A.data_ptr(), lda, A.stride(0),
                                         B.data_ptr(), ldb, B.stride(0), beta, out.data_ptr(), ldc,
                                         out.stride(0), bp, batch, tA, tB, sp)
        else:
            sgemm_f32_ex(M, N, K, alpha, A.data_ptr(), lda, B.data_ptr(), ldb, beta,
                         out.data_ptr(), ldc, bp, tA, tB, sp)
    else:
        x3 = precision == "tf32x3"
        ws, wsb = scratch((tf32x3_workspace_size if x3 else tf32_workspace_size)(M, N, K, batch))
        if not plain:
            if not x3 or batched:
                raise ValueError("the epilogue is available for single tf32x3 products")
            sgemm_f32_tf32x3_ex(M, N, K, alpha, A.data_ptr(), lda, B.data_ptr(), ldb, beta,
                                out.data_ptr(), ldc, bp, tA, tB, ws, wsb, sp)
        elif batched:
            fn = sgemm_f32_tf32x3_strided_batched if x3 else sgemm_f32_tf32_strided_batched
            fn(M, N, K, A.data_ptr(), lda, A.stride(0), B.data_ptr(), ldb, B.stride(0),
               out.data_ptr(), ldc, out.stride(0), batch, tA, tB, ws, wsb, sp)
        else:
            fn = sgemm_f32_tf32x3 if x3 else sgemm_f32_tf32
            fn(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, tA, tB, ws,
               wsb, sp)
    return out
