"""Helpers for GPU parity tests: upload seeded operands with NaN guard bands,
run one entry point of the C ABI, download and check the guards."""
from __future__ import annotations

import numpy as np

import dense_fp32_matrix_sgemm_gb300 as sg

GUARD = 256   # floats of NaN before and after every device buffer


def _upload(arr: np.ndarray, offset: int):
    import torch
    flat = np.ascontiguousarray(arr).ravel()
    buf = torch.full((2 * GUARD + offset + flat.size,), float("nan"), dtype=torch.float32,
                     device="cuda")
    if flat.size:
        buf[GUARD + offset:GUARD + offset + flat.size] = torch.from_numpy(flat).to("cuda")
    return buf, buf.data_ptr() + 4 * (GUARD + offset)


def tf32x3_planes_bytes(M: int, N: int, K: int, batch: int) -> int:
    """The least workspace of the tf32x3 entry points: the hi and lo planes of
    op(A) and op(B), rows of round_up(K, 32) floats, each operand's region
    rounded up to 256 bytes (no room for the partial tiles of tail tiles
    split in K)."""
    Kp = (K + 31) // 32 * 32
    region = lambda rows: (2 * batch * rows * Kp * 4 + 255) // 256 * 256
    return region(M) + region(N)


def run(case: dict, *, entry: str = "sgemm_f32", offset: int = 0, strideB=None,
        stream=None, splits: int = 0, planes_only: bool = False) -> np.ndarray:
    """Run the case on the GPU; returns C (batch, M, N).

    ``offset`` shifts every buffer by that many floats (4-byte aligned only when
    offset % 4 != 0), exercising the scalar-access path.  ``planes_only`` gives
    a tf32x3 entry only the planes' bytes of workspace (whole-tile schedule).
    Asserts that the guard bands and the padding columns of C are still NaN
    afterwards.
    """
    import torch
    batch, M, N, K = case["batch"], case["M"], case["N"], case["K"]
    lda, ldb, ldc = case["lda"], case["ldb"], case["ldc"]
    Abuf, pA = _upload(case["A"], offset)
    Bsrc = case["B"] if strideB != 0 else case["B"][:1]
    Bbuf, pB = _upload(Bsrc, offset)
    Cbuf, pC = _upload(np.full((batch, M, ldc), np.nan, np.float32), offset)
    sA = case["A"][0].size
    sB = 0 if strideB == 0 else case["B"][0].size
    sC = M * ldc
    s = stream if stream is not None else torch.cuda.current_stream().cuda_stream
    fn = getattr(sg, entry)
    extra = ()
    if entry == "sgemm_f32_streamk":
        need = sg.streamk_workspace_size(M, N, K, case["transA"], case["transB"])
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        extra = (ws.data_ptr(), need)
    if entry == "sgemm_f32_splitk":
        need = sg.splitk_workspace_size(M, N, K, splits)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        extra = (splits, ws.data_ptr(), need)
    if "tf32" in entry:
        size = sg.tf32x3_workspace_size if "tf32x3" in entry else sg.tf32_workspace_size
        need = size(M, N, K, batch)
        if planes_only:
            need = tf32x3_planes_bytes(M, N, K, batch)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        extra = (ws.data_ptr(), need)
    if entry.endswith("strided_batched"):
        fn(M, N, K, pA, lda, sA, pB, ldb, sB, pC, ldc, sC, batch, case["transA"],
           case["transB"], *extra, s)
    else:
        assert batch == 1
        fn(M, N, K, pA, lda, pB, ldb, pC, ldc, case["transA"], case["transB"], *extra, s)
    torch.cuda.synchronize()
    out = Cbuf.cpu().numpy()
    assert np.isnan(out[:GUARD + offset]).all(), "write before the start of C"
    assert np.isnan(out[GUARD + offset + batch * M * ldc:]).all(), "write past the end of C"
    for name, buf in (("A", Abuf), ("B", Bbuf)):
        host = buf.cpu().numpy()
        assert np.isnan(host[:GUARD + offset]).all(), f"{name} guard overwritten"
    C = out[GUARD + offset:GUARD + offset + batch * M * ldc].reshape(batch, M, ldc)
    if ldc > N:
        assert np.isnan(C[:, :, N:]).all(), "padding columns of C were written"
    return C[:, :, :N]
