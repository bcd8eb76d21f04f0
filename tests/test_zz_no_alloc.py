"""sgemm_f32_tf32x3_noalloc: the tensor-core product for callers that cannot
allocate device memory (hosts that own all device memory and forbid
allocation inside their GEMM callback, or loops that cannot afford cudaMalloc).

Every call reuses the same built-in scratch, so each result is checked against
the CPU oracle element by element (the library's FP32 bound), and against what
sgemm_f32_tf32x3 with a caller-supplied workspace gives on the same inputs,
call after call.  This file is collected last on purpose, so a run that stops
at the first failure has already run every other test.
"""
import numpy as np
import pytest

import dense_fp32_matrix_sgemm_gb300 as sg
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _run_both(case):
    import torch
    M, N, K = case["M"], case["N"], case["K"]
    A = torch.from_numpy(case["A"][0]).cuda()
    B = torch.from_numpy(case["B"][0]).cuda()
    C_ref = torch.full((M, case["ldc"]), float("nan"), device="cuda")
    C_new = torch.full((M, case["ldc"]), float("nan"), device="cuda")
    need = sg.tf32x3_workspace_size(M, N, K, 1)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    sg.sgemm_f32_tf32x3(M, N, K, A.data_ptr(), case["lda"], B.data_ptr(), case["ldb"],
                        C_ref.data_ptr(), case["ldc"], case["transA"], case["transB"],
                        ws.data_ptr(), need, s)
    sg.sgemm_f32_tf32x3_noalloc(M, N, K, A.data_ptr(), case["lda"], B.data_ptr(), case["ldb"],
                                C_new.data_ptr(), case["ldc"], case["transA"], case["transB"], s)
    torch.cuda.synchronize()
    return C_ref.cpu().numpy(), C_new.cpu().numpy()


def _check(case):
    M, N, K = case["M"], case["N"], case["K"]
    ref, new = _run_both(case)
    C_or, S = oracle.sgemm(case["A"][0], case["B"][0], M, N, K, transA=case["transA"],
                           transB=case["transB"], lda=case["lda"], ldb=case["ldb"],
                           with_scale=True)
    assert np.isfinite(new[:, :N]).all()
    # against the oracle, element by element
    ok = oracle.within_tolerance(new[:, :N], C_or, S)
    assert ok.all(), f"{int((~ok).sum())} outputs outside the bound against the oracle"
    # and the workspace entry point on the same inputs gives the same bits: the
    # two differ only in where the split operands live
    assert np.array_equal(new[:, :N], ref[:, :N]), "differs from sgemm_f32_tf32x3"
    if case["ldc"] > N:
        assert np.isnan(new[:, N:]).all(), "padding columns of C were written"


def test_noalloc_matches_oracle_two_calls_in_a_row():
    # two different problems back to back: the second call must not see
    # anything the first one left in the shared scratch
    cases = [workloads.make_operands(1000, 600, 700, transA=1, dist="normal", seed=11, key=400),
             workloads.make_operands(513, 1023, 1024, transB=1, ldc=1028, dist="uniform",
                                     seed=12, key=401)]
    for case in cases:
        _check(case)
    assert sg.device_status(reset=True) == 0


def test_noalloc_at_the_scratch_limit():
    # 2048^3 needs exactly the 64 MiB of scratch: 2 * (2048 + 2048) * 2048 * 4
    cap = sg.tf32x3_noalloc_max_bytes()
    assert sg.tf32x3_workspace_size(2048, 2048, 2048, 1) == cap
    _check(workloads.make_operands(2048, 2048, 2048, dist="uniform", seed=13, key=402))
    assert sg.device_status(reset=True) == 0


def test_noalloc_when_only_the_planes_fit():
    # 72 tiles of 128 x 128 on 152 SMs: with a full workspace each is split
    # into two K segments, whose partial tiles (9.4 MB) do not fit beside
    # these planes (63.75 MiB) in the scratch, so the call computes whole
    # tiles; on small integers both schedules are exact, hence equal
    cap = sg.tf32x3_noalloc_max_bytes()
    M, N, K = 1024, 1152, 3840
    assert sg.tf32x3_workspace_size(M, N, K, 1) > cap
    _check(workloads.make_operands(M, N, K, dist="int", seed=14, key=403))
    assert sg.device_status(reset=True) == 0


def test_noalloc_rejects_problems_beyond_its_scratch():
    cap = sg.tf32x3_noalloc_max_bytes()
    assert cap == 64 << 20
    # one 32-wide K group past the limit (plane rows are round_up(K, 32) floats)
    M, N, K = 2048, 2048, 2052
    assert sg.tf32x3_workspace_size(M, N, K, 1) > cap
    st = sg.sgemm_f32_tf32x3_noalloc(M, N, K, 16, K, 16, N, 16, N, 0, 0, 0, check=False)
    assert st == 8
    assert "built-in scratch" in sg.last_error()
    M = N = K = 4096          # needs 2 * 8192 * 4096 * 4 = 256 MiB
    st = sg.sgemm_f32_tf32x3_noalloc(M, N, K, 16, K, 16, N, 16, N, 0, 0, 0, check=False)
    assert st == 8
