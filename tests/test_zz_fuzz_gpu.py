"""Randomized GPU parity over every computing entry point of the C ABI.

The hand-written cases in test_parity_gpu.py pick shapes one at a time; this
file draws 120 seeded combinations of entry point, shape (tile multiples,
ragged tails, single rows and columns, K = 0), layout (transA, transB), padded
leading dimensions, misaligned base pointers, batch size and value
distribution, and checks each result against the oracle element by element:

  * FP32 paths (CUDA cores, split-K, 3xTF32, with or without the epilogue):
    |C - C_ref| <= 1e-5 * S + 1e-6, S = |alpha| sum_k |a||b| + |beta||C| + |b|;
  * plain TF32: the same bound with 2e-3 in place of 1e-5 (one TF32 rounding,
    2^-11, on each factor of every product, plus margin);
  * small-integer inputs with K * 16 < 2^24 and no scaling: bit-exact.

Every buffer has NaN guard bands and NaN padding columns in C, which must
survive; the device status word must stay clear.  Sizes keep the oracle to a
few seconds in all.
"""
from __future__ import annotations

import numpy as np
import pytest

import dense_fp32_matrix_sgemm_gb300 as sg
import oracle
import workloads

from gpu_util import GUARD, run

pytestmark = pytest.mark.gpu

ENTRIES = ["sgemm_f32", "sgemm_f32_strided_batched", "sgemm_f32_splitk", "sgemm_f32_ex",
           "sgemm_f32_ex_strided_batched", "sgemm_f32_tf32x3", "sgemm_f32_tf32x3_strided_batched",
           "sgemm_f32_tf32x3_ex", "sgemm_f32_tf32", "sgemm_f32_tf32_strided_batched"]
TF32_REL = 2e-3
NCASES = 120


def _dim(rng, hi):
    """A size in 1..hi: mostly ragged, sometimes a multiple of the 128 tile, sometimes tiny."""
    r = rng.random()
    if r < 0.2:
        return int(rng.integers(1, 9))
    if r < 0.35:
        return int(min(hi, 128 * rng.integers(1, max(2, hi // 128 + 1))))
    return int(rng.integers(1, hi + 1))


def _draw_cases():
    rng = np.random.default_rng(20261202)
    cases = []
    for i in range(NCASES):
        entry = ENTRIES[i % len(ENTRIES)]
        ex = "_ex" in entry
        big = 300 if ex else 700
        c = dict(entry=entry, key=3000 + i, seed=int(rng.integers(1 << 30)))
        c["M"], c["N"] = _dim(rng, big), _dim(rng, big)
        if entry == "sgemm_f32_splitk":
            c["M"], c["N"] = _dim(rng, 260), _dim(rng, 260)
            c["K"] = int(rng.integers(1, 6000))
            c["splits"] = int(rng.choice([0, 0, 2, 3, 7, 64]))
        else:
            c["K"] = 0 if rng.random() < 0.04 else _dim(rng, 1200 if not ex else 400)
        c["batch"] = int(rng.integers(1, 4)) if entry.endswith("strided_batched") else 1
        c["transA"], c["transB"] = int(rng.integers(2)), int(rng.integers(2))
        c["pads"] = [int(rng.choice([0, 0, 1, 3, 4, 7])) for _ in range(3)]
        c["offset"] = int(rng.choice([0, 0, 0, 1, 2, 3]))
        c["dist"] = str(rng.choice(["uniform", "uniform", "normal", "int"]))
        if ex:
            c["alpha"] = float(rng.choice([1.0, 0.0, -0.75, 2.5]))
            c["beta"] = float(rng.choice([0.0, 1.0, -1.25, 0.5]))
            c["bias"] = bool(rng.integers(2))
        cases.append(c)
    return cases


CASES = _draw_cases()


def _operands(c):
    M, N, K, batch = c["M"], c["N"], c["K"], c["batch"]
    pa, pb, pc = c["pads"]
    lda = (M if c["transA"] else K) + pa
    ldb = (K if c["transB"] else N) + pb
    return workloads.make_operands(M, N, K, batch=batch, transA=c["transA"],
                                   transB=c["transB"], lda=max(lda, 1), ldb=max(ldb, 1),
                                   ldc=N + pc, dist=c["dist"], seed=c["seed"], key=c["key"])


def _guarded(arr, offset):
    import torch
    flat = np.ascontiguousarray(arr, dtype=np.float32).ravel()
    buf = torch.full((2 * GUARD + offset + flat.size,), float("nan"), device="cuda")
    if flat.size:
        buf[GUARD + offset:GUARD + offset + flat.size] = torch.from_numpy(flat).cuda()
    return buf, buf.data_ptr() + 4 * (GUARD + offset)


def _run_ex(case, c, C_in, bias):
    """sgemm_f32_ex / _strided_batched / sgemm_f32_tf32x3_ex with guard bands."""
    import torch
    M, N, K, batch = case["M"], case["N"], case["K"], case["batch"]
    lda, ldb, ldc = case["lda"], case["ldb"], case["ldc"]
    off = c["offset"]
    Cfull = np.full((batch, M, ldc), np.nan, np.float32)
    if C_in is not None:
        Cfull[:, :, :N] = C_in
    Abuf, pA = _guarded(case["A"], off)
    Bbuf, pB = _guarded(case["B"], off)
    Cbuf, pC = _guarded(Cfull, off)
    if bias is not None:
        bbuf, pbias = _guarded(bias, 0)
    else:
        pbias = 0
    s = torch.cuda.current_stream().cuda_stream
    a, b, tA, tB = c["alpha"], c["beta"], case["transA"], case["transB"]
    if c["entry"] == "sgemm_f32_ex":
        sg.sgemm_f32_ex(M, N, K, a, pA, lda, pB, ldb, b, pC, ldc, pbias, tA, tB, s)
    elif c["entry"] == "sgemm_f32_ex_strided_batched":
        sg.sgemm_f32_ex_strided_batched(M, N, K, a, pA, lda, case["A"][0].size, pB, ldb,
                                        case["B"][0].size, b, pC, ldc, M * ldc, pbias, batch,
                                        tA, tB, s)
    else:
        need = sg.tf32x3_workspace_size(M, N, K, 1)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device="cuda")
        sg.sgemm_f32_tf32x3_ex(M, N, K, a, pA, lda, pB, ldb, b, pC, ldc, pbias, tA, tB,
                               ws.data_ptr(), need, s)
    torch.cuda.synchronize()
    out = Cbuf.cpu().numpy()
    n = batch * M * ldc
    assert np.isnan(out[:GUARD + off]).all(), "write before the start of C"
    assert np.isnan(out[GUARD + off + n:]).all(), "write past the end of C"
    for name, buf in (("A", Abuf), ("B", Bbuf)):
        assert np.isnan(buf.cpu().numpy()[:GUARD + off]).all(), f"{name} guard overwritten"
    C = out[GUARD + off:GUARD + off + n].reshape(batch, M, ldc)
    if ldc > N:
        assert np.isnan(C[:, :, N:]).all(), "padding columns of C were written"
    return C[:, :, :N]


def _label(c):
    keys = ("entry", "M", "N", "K", "batch", "transA", "transB", "pads", "offset", "dist",
            "splits", "alpha", "beta", "bias")
    return " ".join(f"{k}={c[k]}" for k in keys if k in c)


@pytest.mark.parametrize("idx", range(NCASES))
def test_random_case(idx):
    c = CASES[idx]
    label = _label(c)
    case = _operands(c)
    M, N, K, batch = case["M"], case["N"], case["K"], case["batch"]
    assert sg.device_status(reset=True) == 0
    rel = TF32_REL if c["entry"] in ("sgemm_f32_tf32", "sgemm_f32_tf32_strided_batched") else \
        oracle.REL_TOL
    exact = c["dist"] == "int" and K * 16 < (1 << 24)

    if "_ex" in c["entry"]:
        rng = np.random.default_rng(c["seed"] + 1)
        C_in = rng.standard_normal((batch, M, N)).astype(np.float32) if c["beta"] != 0.0 else None
        bias = rng.standard_normal(N).astype(np.float32) if c["bias"] else None
        got = _run_ex(case, c, C_in, bias)
        exact = False
        refs, scales = [], []
        for z in range(batch):
            r, s = oracle.sgemm_ex(case["A"][z], case["B"][z], M, N, K, alpha=c["alpha"],
                                   beta=c["beta"], C_in=C_in[z] if C_in is not None else None,
                                   bias=bias, transA=case["transA"], transB=case["transB"],
                                   lda=case["lda"], ldb=case["ldb"])
            refs.append(r)
            scales.append(s)
        ref, S = np.stack(refs), np.stack(scales)
    else:
        got = run(case, entry=c["entry"], offset=c["offset"], splits=c.get("splits", 0))
        if batch == 1:
            ref, S = oracle.sgemm(case["A"][0], case["B"][0], M, N, K, transA=case["transA"],
                                  transB=case["transB"], lda=case["lda"], ldb=case["ldb"],
                                  with_scale=True)
            ref, S = ref[None], S[None]
        else:
            ref, S = oracle.sgemm_strided_batched(case["A"], case["B"], M, N, K, batch,
                                                  transA=case["transA"], transB=case["transB"],
                                                  lda=case["lda"], ldb=case["ldb"],
                                                  with_scale=True)

    assert sg.device_status(reset=True) == 0, f"{label}: device status set"
    assert np.isfinite(got).all(), f"{label}: non-finite outputs"
    if exact:
        bad = got != ref
        assert not bad.any(), f"{label}: {int(bad.sum())} outputs differ from the exact result"
    ok = oracle.within_tolerance(got, ref, S, rel=rel)
    if not ok.all():
        idx_bad = np.argwhere(~ok)[:5]
        raise AssertionError(f"{label}: {int((~ok).sum())} outputs outside the bound, first "
                             f"{idx_bad.tolist()} got {got[~ok][:5]} want {ref[~ok][:5]}")


# sgemm_f32_streamk: sizes large enough that the entry's choices all occur:
# a K-contiguous operand turned into a workspace copy (2MNK >= 1.6e10), the
# TMA kernel or the cp.async kernel (alignment), stream-K below four waves of
# two CTAs per SM and the plain grid above, pieces of one or two K slices.
NSTREAMK = 24


def _draw_streamk_cases():
    rng = np.random.default_rng(20261203)
    cases = []
    for i in range(NSTREAMK):
        c = dict(entry="sgemm_f32_streamk", key=5000 + i, seed=int(rng.integers(1 << 30)))
        c["M"] = int(rng.integers(1000, 3600))
        c["N"] = int(rng.integers(1000, 3600))
        c["K"] = int(rng.choice([int(rng.integers(1, 64)), int(rng.integers(64, 2600))]))
        c["batch"] = 1
        c["transA"], c["transB"] = int(rng.integers(2)), int(rng.integers(2))
        # most cases 16-byte aligned (the TMA kernels), the rest not (cp.async)
        dims = [c["M"] if c["transA"] else c["K"], c["K"] if c["transB"] else c["N"], c["N"]]
        if rng.random() < 0.6:
            c["pads"] = [int((-d) % 4 + 4 * rng.integers(0, 2)) for d in dims]
            c["offset"] = 0
        else:
            c["pads"] = [int(rng.choice([0, 1, 3])) for _ in dims]
            c["offset"] = int(rng.choice([0, 1]))
        c["dist"] = str(rng.choice(["uniform", "normal", "int"]))
        cases.append(c)
    return cases


STREAMK_CASES = _draw_streamk_cases()


@pytest.mark.parametrize("idx", range(NSTREAMK))
def test_random_streamk_case(idx):
    c = STREAMK_CASES[idx]
    label = _label(c)
    case = _operands(c)
    M, N, K = case["M"], case["N"], case["K"]
    assert sg.device_status(reset=True) == 0
    got = run(case, entry="sgemm_f32_streamk", offset=c["offset"])
    assert sg.device_status(reset=True) == 0, f"{label}: device status set"
    ref, S = oracle.sgemm(case["A"][0], case["B"][0], M, N, K, transA=case["transA"],
                          transB=case["transB"], lda=case["lda"], ldb=case["ldb"],
                          with_scale=True)
    assert np.isfinite(got).all(), f"{label}: non-finite outputs"
    if c["dist"] == "int" and K * 16 < (1 << 24):
        bad = got[0] != ref
        assert not bad.any(), f"{label}: {int(bad.sum())} outputs differ from the exact result"
    ok = oracle.within_tolerance(got[0], ref, S)
    assert ok.all(), f"{label}: {int((~ok).sum())} outputs outside the bound"
