#!/usr/bin/env python3
"""Benchmark: SGEMM TFLOP/s and fraction of the GB300 FP32 peak at 3072^3.

One step = one C = A B call (M = N = K = 3072, row-major, U[-1,1) inputs)
through the C ABI, inputs already resident in HBM.  Three input sets rotate
(3 x 113 MB > 129 MB L2) so every step starts with its operands out of L2.
Each step is timed with CUDA events on the stream the kernel is launched on;
the timed region is bracketed by a barrier and a device synchronisation.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead (the
only other place this script executes the oracle), on a bounded row sample of
the same workload.

Multi-GPU: the GEMM does not need a collective; with N ranks each GPU runs
an independent replica (weak scaling) and the value is the sum over ranks
(total FLOPs / max time over ranks).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

WORKLOAD = "sgemm_3072x3072x3072_uniform"
METRIC = "SGEMM TFLOP/s and % of GB300 FP32 peak at 3072³ (1 GPU), vs CPU oracle"
FP32_LANES_PER_SM = 128          # FP32 FMA units per Blackwell SM
TF32_PER_BF16 = 1.1 / 2.25       # nominal dense TF32 / BF16 tensor rates of GB300
SM_MAX_MHZ_DEFAULT = 2070.0
ROTATING_SETS = 3


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=WORKLOAD, choices=sorted(workloads.WORKLOADS))
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="target CPU time of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-tf32x3", action="store_true", help="skip the tensor-core path report")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the per-workload table (every named workload, both FP32 paths)")
    p.add_argument("--raster-group", type=int, default=0,
                   help="tile rows per raster group for every call (sgemm_set_raster_group; "
                        "0 = the library's 8): for L2 measurements of the block order")
    p.add_argument("--tf32x3-chunk-k", type=int, default=0,
                   help="K per chunk of the 3xTF32 K-chunked kernel for every call "
                        "(sgemm_set_tf32x3_chunk_k; 0 = the library's 128)")
    p.add_argument("--tc-only", action="store_true",
                   help="time only sgemm_f32_tf32x3 on the workload (W warm-up, K timed calls) "
                        "and print one JSON object with its RRMSE against the oracle")
    p.add_argument("--plain-only", action="store_true",
                   help="time only plain sgemm_f32 on the workload (W warm-up, K timed calls) and "
                        "print one JSON object of that measurement, not the bench line")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank scalar over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tflops(flops_per_step: float, steps: int, max_total_ms: float, world: int) -> float:
    """Whole-job throughput of `world` replicas: every rank ran `steps` steps of
    `flops_per_step`, the job took as long as the slowest rank."""
    return world * flops_per_step * steps / (max_total_ms * 1e-3) / 1e12


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open("/tmp/_sgemm_clocks_%d.csv" % os.getpid(), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.out:
            self.out.close()

    def summary(self):
        path = "/tmp/_sgemm_clocks_%d.csv" % os.getpid()
        if self.proc is None or not os.path.exists(path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        for line in open(path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        os.unlink(path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, parts in rows:
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [r[0] for r in rows]
        power = []
        for _, _, parts in rows:
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "sm_mhz_min": min(loaded), "samples": len(rows),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


# ------------------------------------------------------------------ helpers

KERNEL_SOURCES = {
    "sgemm_simt_kernel": ["gemm_args.h", "device_utils.cuh", "simt_sgemm.cuh", "simt_launch.cuh",
                          "simt_nn.cu"],
    "tf32x3_persistent_kernel": ["gemm_args.h", "tc_utils.cuh", "tf32x3.cu"],
    "tf32x3_chunked_kernel": ["gemm_args.h", "tc_utils.cuh", "tf32x3.cu"],
    "sgemm_simt_streamk_kernel": ["gemm_args.h", "device_utils.cuh", "simt_sgemm.cuh",
                                  "simt_launch.cuh", "simt_tn.cu"],
    "sgemm_simt_streamk_tma_kernel": ["gemm_args.h", "device_utils.cuh", "simt_sgemm.cuh",
                                      "simt_launch.cuh", "tc_utils.cuh", "simt_tma.cu"],
    "sgemm_simt_tma_kernel": ["gemm_args.h", "device_utils.cuh", "simt_sgemm.cuh",
                              "simt_launch.cuh", "tc_utils.cuh", "simt_tma.cu"],
}


def kernel_source_hash(kernel: str = "sgemm_simt_kernel") -> str:
    """Hash of the sources that make up a kernel; profiles record it so a stale
    DRAM-traffic figure is never reported for a changed kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_fp32_matrix_sgemm_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """Bytes per launch (dram read + write) from the committed ncu summary, if it
    was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash(kernel)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#") and parts[0] == kernel \
                and parts[1] == workload and parts[2] == want:
            return int(parts[3])
    return None


def simt_kernel_label(M, N, batch, transB, sms, K=3072, transA=0):
    """The kernel the library's launcher picks for 16-byte aligned operands
    (same rules as csrc/simt_launch.cuh and csrc/simt_tma.cu): problems whose
    128x128 tiles cover at most half the SMs split K over a cluster; row-major
    B, or both operands stored transposed, take the TMA-fed kernel (persistent
    for short reductions with A stored transposed and row-major B); row-major
    A with B stored transposed takes the cp.async kernel at two CTAs per SM."""
    tiles = batch * -(-M // 128) * -(-N // 128)
    if tiles * 2 <= sms and K > 32:
        return "sgemm_simt_kernel 128x128 tile, K split over the CTAs of a cluster"
    if transA or not transB:
        if transB:
            a = "A stored transposed, B^T as 128-byte-swizzled K boxes"
        else:
            a = "A stored transposed" if transA else "row-major A as 128-byte-swizzled K boxes"
        if transA and not transB and K <= 256 and tiles >= 4 * sms:
            return ("sgemm_simt_persist_tma_kernel 128x128 tile, BK 32, 3 stages, 2 CTAs/SM, "
                    f"TMA-fed ({a}), loads across tile boundaries, fma.rn.f32x2")
        return ("sgemm_simt_tma_kernel 128x128 tile, BK 32, 3 stages, 2 CTAs/SM, "
                f"TMA-fed ({a}), fma.rn.f32x2")
    return "sgemm_simt_kernel 128x128 tile, BK 32, 2 stages, 2 CTAs/SM, fma.rn.f32x2"


def _chunked_split(tiles, kblocks, sms):
    """K segments per tail tile (csrc/tf32x3.cu chunked_plan), 0 for whole tiles."""
    tail = tiles % sms
    split = min(sms // tail, kblocks // 2) if tail else 0
    return split if split >= 2 else 0


def _chunked_cost_us(tiles, K, kblocks, bn, sms):
    split = _chunked_split(tiles, kblocks, sms)
    tile_us = 0.019 * K * (1.5 if bn == 256 else 1.0)
    if split:
        part = split * (tiles % sms) * 128 * bn * 4
        return (tiles // sms + 1.0 / split) * tile_us + 2.0 * part / 20e6
    return (tiles // sms + (1 if tiles % sms else 0)) * tile_us


def tc_wide_tile(M, N, K, batch, sms):
    """The K-chunked kernel's tile width (csrc/tf32x3.cu, tc_wide_tile and
    chunked_cost_us)."""
    if K <= 256:
        return False
    tm = -(-M // 128)
    wide, narrow = batch * tm * -(-N // 256), batch * tm * -(-N // 128)
    return (_chunked_cost_us(wide, K, -(-K // 16), 256, sms)
            <= _chunked_cost_us(narrow, K, -(-K // 32), 128, sms))


def tc_split_tail(M, N, K, batch, sms):
    """K segments per tail tile of the K-chunked kernel (csrc/tf32x3.cu,
    chunked_plan), 0 when the tiles run whole: the last wave's tiles are split
    into SMs // tail segments of at least two K blocks when that is two or
    more (the workspace has room for their partial tiles)."""
    if K <= 256:
        return 0
    wide = tc_wide_tile(M, N, K, batch, sms)
    bn, bk = (256, 16) if wide else (128, 32)
    return _chunked_split(batch * -(-M // 128) * -(-N // bn), -(-K // bk), sms)


def tc_plan(M, N, K, batch, transA, transB, aligned=True, rows128=True, sms=152):
    """(kernels label, launches) of one 3xTF32 call, mirroring csrc/tf32x3.cu:
    a K-contiguous operand (row-major A, B stored transposed) with aligned
    rows (16 bytes for K <= 256, 128 bytes beyond: `aligned`, `rows128`) is
    read as its own hi term; its lo term is made by converter warps inside
    the GEMM when K <= 64, or K <= 256 with at most 8 tiles reading each of
    its panels, else written by the split kernel as a lo plane; other
    operands are split into hi and lo planes.  Tail tiles split in K add the
    fix-up kernel."""
    tiles_m, tiles_n = -(-M // 128), -(-N // 128)   # K <= 256 takes 128-wide tiles

    def conv(reuse):
        return K <= 64 or (K <= 256 and reuse <= 8)
    ok = aligned if K <= 256 else aligned and rows128
    parts, split = [], []
    for name, kcontig, reuse in (("A", not transA, tiles_n), ("B", bool(transB), tiles_m)):
        if kcontig and ok:
            if conv(reuse):
                parts.append(f"{name} raw, lo by converter warps")
            else:
                parts.append(f"{name} raw as hi")
                split.append(f"{name} lo plane")
        else:
            split.append(f"{name} hi/lo planes")
    if K <= 256:
        gemm = ("tf32x3_persistent_kernel (one CTA per SM; 128x128 tiles; TMA ring, tcgen05 "
                "kind::tf32, TMEM, TMA-store epilogue" +
                ("; " + ", ".join(parts) if parts else "") + ")")
    else:
        width = "128x256" if tc_wide_tile(M, N, K, batch, sms) else "128x128"
        gemm = (f"tf32x3_chunked_kernel (one CTA per SM; {width} tiles; "
                "TMA ring, tcgen05 kind::tf32 into two TMEM chunk accumulators, each 128 of K "
                "added into fp32 registers by 8 epilogue warps, TMA-store epilogue" +
                ("; " + ", ".join(parts) if parts else "") + ")")
    launches = 1
    nseg = tc_split_tail(M, N, K, batch, sms)
    if nseg:
        gemm += (f", last wave's tiles split into {nseg} K segments + tf32x3_fixup_kernel "
                 "(adds the segments' partial tiles)")
        launches += 1
    if split:
        return f"split_kernel ({', '.join(split)}) + {gemm}", launches + 1
    return gemm, launches


def tc_kernel_name(K: int) -> str:
    """The 3xTF32 GEMM kernel csrc/tf32x3.cu runs for reduction depth K: the
    single-pass persistent kernel up to K = 256, the K-chunked one beyond."""
    return "tf32x3_persistent_kernel" if K <= 256 else "tf32x3_chunked_kernel"


def graph_ms(torch, stream, fn, ms_one):
    """Device time per call with the host's launch cost taken out: `reps`
    back-to-back calls captured in one CUDA graph, replayed three times, the
    median replay divided by `reps`."""
    reps = 20 if ms_one < 0.5 else 3
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(reps):
            fn()
    ts = []
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
    return sorted(ts)[1] / reps


def workload_table(torch, sg, dev, stream, sp, reps=5):
    """ms, TFLOP/s and compulsory-byte GB/s of sgemm_f32 and sgemm_f32_tf32x3 on
    every named workload (operands resident on the device, median of `reps`
    after two warm-ups), each call timed alone between CUDA events (the host's
    launch cost included: it dominates the smallest problems), and `*_graph_ms`
    the device time per call from back-to-back calls in a CUDA graph."""
    out = {}
    for name, w in workloads.WORKLOADS.items():
        case = workloads.make_case(w)
        lda, ldb, ldc = case["lda"], case["ldb"], case["ldc"]
        dA = torch.from_numpy(case["A"].reshape(-1)).to(dev)
        dB = torch.from_numpy(case["B"].reshape(-1)).to(dev)
        dC = torch.empty(w.batch * w.M * ldc, dtype=torch.float32, device=dev)
        need = sg.tf32x3_workspace_size(w.M, w.N, w.K, w.batch)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        sA, sB, sC = case["A"][0].size, case["B"][0].size, w.M * ldc
        row = {"M": w.M, "N": w.N, "K": w.K, "batch": w.batch, "transA": w.transA,
               "transB": w.transB, "min_bytes": workloads.min_bytes(w.M, w.N, w.K, w.batch)}

        def simt():
            sg.sgemm_f32_strided_batched(w.M, w.N, w.K, dA.data_ptr(), lda, sA, dB.data_ptr(), ldb,
                                         sB, dC.data_ptr(), ldc, sC, w.batch, w.transA, w.transB,
                                         sp)

        def tc():
            sg.sgemm_f32_tf32x3_strided_batched(w.M, w.N, w.K, dA.data_ptr(), lda, sA,
                                                dB.data_ptr(), ldb, sB, dC.data_ptr(), ldc, sC,
                                                w.batch, w.transA, w.transB, ws.data_ptr(), need,
                                                sp)

        legs = [("simt", simt), ("tf32x3", tc)]
        sk_need = sg.streamk_workspace_size(w.M, w.N, w.K, w.transA, w.transB) if w.batch == 1 else 0
        if sk_need:
            sk_ws = torch.empty(sk_need, dtype=torch.uint8, device=dev)

            def streamk():
                sg.sgemm_f32_streamk(w.M, w.N, w.K, dA.data_ptr(), lda, dB.data_ptr(), ldb,
                                     dC.data_ptr(), ldc, w.transA, w.transB, sk_ws.data_ptr(),
                                     sk_need, sp)

            legs.append(("simt_streamk", streamk))
        for label, fn in legs:
            for _ in range(2):
                fn()
            ts = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
            ms = sorted(ts)[len(ts) // 2]
            row[label + "_ms"] = ms
            row[label + "_tflops"] = workloads.flops(w.M, w.N, w.K, w.batch) / (ms * 1e-3) / 1e12
            gms = graph_ms(torch, stream, fn, ms)
            row[label + "_graph_ms"] = gms
            row[label + "_graph_tflops"] = workloads.flops(w.M, w.N, w.K, w.batch) / (gms * 1e-3) / 1e12
            # compulsory bytes / time: the figure that matters where a path
            # is bandwidth-bound (the batched QK^T shape on the tensor cores)
            row[label + "_gbs"] = row["min_bytes"] / (ms * 1e-3) / 1e9
        out[name] = row
        del dA, dB, dC, ws
        if sk_need:
            del sk_ws
    torch.cuda.empty_cache()
    return out


def tf32_probe_tflops(torch, sg, dev, stream, iters=16384, reps=5):
    """Measured TF32 tensor-pipe peak: the library's tcgen05.mma probe (one CTA
    per SM, operands in shared memory), CUDA events, median of `reps`."""
    out = torch.empty(sg.probe_out_elems(), dtype=torch.float32, device=dev)
    sp = stream.cuda_stream
    sg.probe_tf32_mma(256, out.data_ptr(), sp)
    ts, flops = [], 0.0
    for _ in range(reps):
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        flops = sg.probe_tf32_mma(iters, out.data_ptr(), sp)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ts.append(e0.elapsed_time(e1))
    ms = sorted(ts)[len(ts) // 2]
    return flops / (ms * 1e-3) / 1e12


def streamk_plan(M, N, K, transA, transB, sms, aligned=True):
    """(transposes, stream-K used, tile kernel) of one sgemm_f32_streamk call:
    a transpose per turned operand, then the tile kernel, plus the fix-up pass
    when stream-K applies.  Mirrors the library's rule (include/sgemm_gb300.h,
    csrc/api.cu): in problems with 2MNK >= 1.6e10, row-major A is turned when
    N >= 1024 and B^T when M >= 1024 (the copies are 16-byte aligned).  Then A
    stored transposed with row-major B takes the TMA-fed kernel when aligned:
    128 x 128 tiles, G = 2 CTAs per SM, stream-K when G < tiles < 4G and the
    tiles do not fill whole waves.  Aligned row-major A that is not turned, or
    both operands stored transposed and neither turned, run the TMA kernel
    directly, without stream-K."""
    big = 2.0 * M * N * K >= 1.6e10
    turn_a = big and not transA and N >= 1024
    turn_b = big and transB and M >= 1024
    tA, tB = bool(transA or turn_a), bool(transB and not turn_b)
    aligned = aligned or (turn_a or turn_b)
    kslices = -(-K // 32)
    if tA and not tB and aligned:
        G = 2 * sms
        tiles = -(-M // 128) * -(-N // 128)
        sk = G < tiles < 4 * G and tiles % G != 0 and kslices >= 2
        kernel = "sgemm_simt_streamk_tma_kernel" if sk else "sgemm_simt_tma_kernel"
    elif tA and not tB:
        tiles = -(-M // 128) * -(-N // 128)
        sk = tiles > sms and tiles % sms != 0 and kslices >= 2
        kernel = "sgemm_simt_streamk_kernel" if sk else "sgemm_simt_kernel"
    elif (tA or not tB) and aligned:   # read directly by the TMA kernel, no stream-K
        sk, kernel = False, "sgemm_simt_tma_kernel"
    else:
        sk, kernel = False, "sgemm_simt_kernel"
    return int(turn_a) + int(turn_b), sk, kernel


def streamk_launches(M, N, K, transA, transB, sms, aligned=True) -> int:
    turned, sk, _ = streamk_plan(M, N, K, transA, transB, sms, aligned)
    return turned + 1 + int(sk)


def step_kernel_label(M, N, K, transA, transB, sms, batch, plain_label, aligned=True) -> str:
    if batch != 1:
        return plain_label
    turned, sk, kernel = streamk_plan(M, N, K, transA, transB, sms, aligned)
    parts = ["transpose_kernel (K-contiguous operand -> workspace copy)"] * turned
    if sk:
        parts.append(f"{kernel} (whole-wave tiles, then one stream-K range per CTA; TMA-fed, "
                     "two CTAs per SM) + streamk_fixup_kernel")
    elif kernel == "sgemm_simt_tma_kernel":
        big = 2.0 * M * N * K >= 1.6e10
        tA = bool(transA or (big and N >= 1024))
        tB = bool(transB and not (big and M >= 1024))
        parts.append(simt_kernel_label(M, N, batch, int(tB), sms, K, int(tA)))
    else:
        parts.append(plain_label)
    return " + ".join(parts)


def cpu_baseline(case, target_s: float):
    """Time the oracle as it stands on a bounded sample of rows of the workload."""
    import oracle
    M, N, K = case["M"], case["N"], case["K"]
    threads = oracle.default_threads()
    A = case["A"][0]
    B = case["B"][0]

    def rows_run(r):
        sub = np.ascontiguousarray(A[:r])
        t = time.perf_counter()
        oracle.sgemm(sub, B, r, N, K, lda=case["lda"], ldb=case["ldb"], nthreads=threads)
        return time.perf_counter() - t

    probe = min(M, max(threads, 32))
    t = rows_run(probe)
    rows = int(min(M, max(probe, probe * target_s / max(t, 1e-6))))
    t = rows_run(rows)
    flops = 2.0 * rows * N * K
    return {"value": flops / t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{rows} of {M} rows of the {M}x{N}x{K} product "
                      f"({flops / 1e9:.1f} GFLOP, {t:.2f} s, fp64 accumulation)",
            "seconds": t}


def cpu_baseline_workloads(target_s: float):
    """The oracle as it stands on every named workload: the whole product when
    it takes under about `target_s`, else its first rows (op(A) rows of any
    layout), the rate then standing for the full product ("extrapolated")."""
    import oracle
    threads = oracle.default_threads()
    out = {}
    for name, w in workloads.WORKLOADS.items():
        case = workloads.make_case(w)
        M, N, K, batch = w.M, w.N, w.K, w.batch
        A, B = case["A"], case["B"]

        def run(rows):
            t = time.perf_counter()
            if batch == 1:
                oracle.sgemm(A[0], B[0], rows, N, K, transA=w.transA, transB=w.transB,
                             lda=case["lda"], ldb=case["ldb"], nthreads=threads)
            else:
                oracle.sgemm_strided_batched(A, B, rows, N, K, batch, transA=w.transA,
                                             transB=w.transB, lda=case["lda"], ldb=case["ldb"],
                                             strideA=A[0].size, strideB=B[0].size,
                                             nthreads=threads)
            return time.perf_counter() - t

        probe = min(M, max(threads, 32))
        t = run(probe)
        rows = int(min(M, max(probe, probe * target_s / max(t, 1e-6))))
        if rows != probe:
            t = run(rows)
        flops = 2.0 * rows * N * K * batch
        out[name] = {"gflops": flops / t / 1e9, "rows": rows, "of_rows": M, "seconds": t,
                     "extrapolated": rows < M,
                     "full_product_s": workloads.flops(M, N, K, batch) / (flops / t)}
        del case, A, B
    return out


# ------------------------------------------------------------------ reference arm

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = workloads.get(args.workload)
    case = workloads.make_case(w)
    M, N, K = w.M, w.N, w.K
    threads = oracle.default_threads()
    # each step: a row slice sized to roughly 0.2 s on this host
    A, B = case["A"][0], case["B"][0]
    t = time.perf_counter()
    oracle.sgemm(np.ascontiguousarray(A[:threads]), B, threads, N, K, nthreads=threads)
    per_row = (time.perf_counter() - t) / threads
    rows = int(max(threads, min(M, 0.2 / max(per_row, 1e-9))))
    sub = np.ascontiguousarray(A[:rows])
    for _ in range(args.warmup):
        oracle.sgemm(sub, B, rows, N, K, nthreads=threads)
    times = []
    for _ in range(args.steps):
        t = time.perf_counter()
        oracle.sgemm(sub, B, rows, N, K, nthreads=threads)
        times.append(time.perf_counter() - t)
    total = sum(times)
    flops = 2.0 * rows * N * K
    value = flops * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64-accumulate", "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"{rows} of {M} rows per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    import dense_fp32_matrix_sgemm_gb300 as sg

    rank, world, local = dist_env()
    if world != args.gpus:
        if world == 1 and args.gpus > 1:
            raise SystemExit("--gpus > 1 must be launched with torch.distributed.run")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    if args.raster_group:
        sg.set_raster_group(args.raster_group)
    if args.tf32x3_chunk_k:
        sg.set_tf32x3_chunk_k(args.tf32x3_chunk_k)
    w = workloads.get(args.workload)
    case = workloads.make_case(w)
    M, N, K, batch = w.M, w.N, w.K, w.batch
    lda, ldb, ldc = case["lda"], case["ldb"], case["ldc"]
    flops = workloads.flops(M, N, K, batch)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream

    # CPU baseline first (rank 0, before any heavy GPU work; no fork involved)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, args.cpu_seconds)
        if not args.no_workloads:
            cpu["per_workload"] = cpu_baseline_workloads(0.3)

    nsets = ROTATING_SETS
    with torch.cuda.stream(stream):
        hA = torch.from_numpy(case["A"].reshape(-1))
        hB = torch.from_numpy(case["B"].reshape(-1))
        sets = []
        for _ in range(nsets):
            dA = hA.to(dev, non_blocking=False).clone()
            dB = hB.to(dev, non_blocking=False).clone()
            dC = torch.empty(batch * M * ldc, dtype=torch.float32, device=dev)
            sets.append((dA, dB, dC))
    torch.cuda.synchronize(dev)

    # The step is one sgemm_f32_streamk call (single problems): the library's
    # fastest FP32 CUDA-core path, with its workspace allocated once here.
    # Batched problems use sgemm_f32_strided_batched.  Plain sgemm_f32 is
    # timed the same way afterwards and reported beside it.
    sk_need = sg.streamk_workspace_size(M, N, K, w.transA, w.transB) if batch == 1 else 0
    sk_ws = torch.empty(max(sk_need, 1), dtype=torch.uint8, device=dev)
    sms_dev = torch.cuda.get_device_properties(dev).multi_processor_count
    aligned = lda % 4 == 0 and ldb % 4 == 0 and ldc % 4 == 0
    rows128 = lda % 32 == 0 and ldb % 32 == 0   # (device buffers are 512-byte aligned)
    launches = (streamk_launches(M, N, K, w.transA, w.transB, sms_dev, aligned) if batch == 1
                else 1)

    def plain_step(i):
        dA, dB, dC = sets[i % nsets]
        if batch == 1:
            sg.sgemm_f32(M, N, K, dA.data_ptr(), lda, dB.data_ptr(), ldb, dC.data_ptr(), ldc,
                         w.transA, w.transB, sp)
        else:
            sg.sgemm_f32_strided_batched(M, N, K, dA.data_ptr(), lda, case["A"][0].size,
                                         dB.data_ptr(), ldb, case["B"][0].size, dC.data_ptr(),
                                         ldc, M * ldc, batch, w.transA, w.transB, sp)

    if args.tc_only:
        need = sg.tf32x3_workspace_size(M, N, K, batch)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)

        def tc_call(i):
            dA, dB, dC = sets[i % nsets]
            sg.sgemm_f32_tf32x3_strided_batched(
                M, N, K, dA.data_ptr(), lda, case["A"][0].size, dB.data_ptr(), ldb,
                case["B"][0].size, dC.data_ptr(), ldc, M * ldc, batch, w.transA, w.transB,
                ws.data_ptr(), need, sp)
        for i in range(args.warmup):
            tc_call(i)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            tc_call(i)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ts = sorted(a.elapsed_time(b) for a, b in ev)
        ms = ts[len(ts) // 2]
        out = {"mode": "tc_only", "entry": "sgemm_f32_tf32x3", "workload": args.workload,
               "chunk_k": args.tf32x3_chunk_k or 128, "steps": args.steps, "median_ms": ms,
               "tflops": flops / (ms * 1e-3) / 1e12}
        if rank == 0 and batch == 1 and not w.transA:
            import oracle
            dC = sets[(args.steps - 1) % nsets][2]
            rows = np.arange(0, M, max(1, M // 256))
            got = dC.view(M, ldc)[rows, :N].cpu().numpy()
            ref = oracle.sgemm(np.ascontiguousarray(case["A"][0][rows]), case["B"][0], len(rows),
                               N, K, lda=lda, ldb=ldb)
            out["rrmse_vs_oracle_256_rows"] = oracle.rrmse(got, ref)
        if rank == 0:
            print(json.dumps(out))
        return

    if args.plain_only:
        # one kernel family, nothing else launched: the form the L2 / raster
        # captures of profiles/ use
        for i in range(args.warmup):
            plain_step(i)
        torch.cuda.synchronize(dev)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i, (a, b) in enumerate(ev):
            a.record(stream)
            plain_step(i)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ts = sorted(a.elapsed_time(b) for a, b in ev)
        ms = ts[len(ts) // 2]
        if rank == 0:
            print(json.dumps({"mode": "plain_only", "entry": "sgemm_f32", "workload": args.workload,
                              "raster_group": args.raster_group or 8, "steps": args.steps,
                              "median_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                              "kernel": simt_kernel_label(M, N, batch, w.transB, sms_dev, K,
                                                          w.transA)}))
        return

    def step(i):
        if batch != 1:
            return plain_step(i)
        dA, dB, dC = sets[i % nsets]
        sg.sgemm_f32_streamk(M, N, K, dA.data_ptr(), lda, dB.data_ptr(), ldb, dC.data_ptr(), ldc,
                             w.transA, w.transB, sk_ws.data_ptr(), sk_need, sp)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        wall0 = time.perf_counter()
        for i in range(args.steps):
            starts[i].record(stream)
            step(i)
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
        wall = time.perf_counter() - wall0
        if world > 1:
            dist.barrier()
    clocks = clk.summary()
    durs = [s.elapsed_time(e) for s, e in zip(starts, ends)]   # ms

    total_ms = reduce_max_over_ranks(sum(durs), dev)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_tflops(flops, args.steps, total_ms, world)

    # end to end through the C ABI from pinned host buffers: every step uploads
    # its A and B, runs the GEMM and downloads C.  Two device buffer sets and
    # three streams (upload, compute, download) let step i+1's upload and step
    # i-1's download overlap step i's GEMM, as a caller streaming matrices would.
    pA = torch.from_numpy(case["A"].reshape(-1)).pin_memory()
    pB = torch.from_numpy(case["B"].reshape(-1)).pin_memory()
    pC = [torch.empty(batch * M * ldc, dtype=torch.float32).pin_memory() for _ in range(2)]
    e2e_steps = max(4, min(args.steps, 20))
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(n):
        uploaded = [torch.cuda.Event(), torch.cuda.Event()]
        computed = [torch.cuda.Event(), torch.cuda.Event()]
        downloaded = [None, None]
        for i in range(n):
            b = i % 2
            dA, dB, dC = sets[b]
            with torch.cuda.stream(up):
                if downloaded[b] is not None:
                    up.wait_event(downloaded[b])      # buffer b's previous result is home
                dA.copy_(pA, non_blocking=True)
                dB.copy_(pB, non_blocking=True)
                uploaded[b].record(up)
            stream.wait_event(uploaded[b])
            step(b)
            computed[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                pC[b].copy_(dC, non_blocking=True)
                downloaded[b] = torch.cuda.Event()
                downloaded[b].record(down)
        for d in downloaded:
            if d is not None:
                stream.wait_event(d)

    e2e_run(2)
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    up.wait_event(e0)
    down.wait_event(e0)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = reduce_max_over_ranks(e0.elapsed_time(e1), dev) / e2e_steps

    # cold L2: the same call after writing a 512 MiB buffer on the same stream
    # before each step (the flush sits outside the events around the call)
    flush = torch.empty(512 * 2**20 // 4, dtype=torch.float32, device=dev)
    cold_steps = max(5, min(args.steps, 20))
    c0 = [torch.cuda.Event(enable_timing=True) for _ in range(cold_steps)]
    c1 = [torch.cuda.Event(enable_timing=True) for _ in range(cold_steps)]
    for i in range(cold_steps):
        with torch.cuda.stream(stream):
            flush.fill_(float(i))
        c0[i].record(stream)
        step(i)
        c1[i].record(stream)
    torch.cuda.synchronize(dev)
    cold = sorted(a.elapsed_time(b) for a, b in zip(c0, c1))
    del flush

    # plain sgemm_f32 (one kernel), same protocol, reported beside the step
    plain_ms = None
    if batch == 1:
        for i in range(args.warmup):
            plain_step(i)
        torch.cuda.synchronize(dev)
        p0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        p1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            p0[i].record(stream)
            plain_step(i)
            p1[i].record(stream)
        torch.cuda.synchronize(dev)
        plain_ms = reduce_max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(p0, p1)), dev) / args.steps
    h2d = (case["A"].size + case["B"].size) * 4
    d2h = batch * M * ldc * 4

    # the tensor-core 3xTF32 path, reported separately on the same inputs
    tc = None
    if not args.no_tf32x3:
        need = sg.tf32x3_workspace_size(M, N, K, batch)
        ws = torch.empty(need, dtype=torch.uint8, device=dev)

        def tc_step(i):
            dA, dB, dC = sets[i % nsets]
            if batch == 1:
                sg.sgemm_f32_tf32x3(M, N, K, dA.data_ptr(), lda, dB.data_ptr(), ldb, dC.data_ptr(),
                                    ldc, w.transA, w.transB, ws.data_ptr(), need, sp)
            else:
                sg.sgemm_f32_tf32x3_strided_batched(
                    M, N, K, dA.data_ptr(), lda, case["A"][0].size, dB.data_ptr(), ldb,
                    case["B"][0].size, dC.data_ptr(), ldc, M * ldc, batch, w.transA, w.transB,
                    ws.data_ptr(), need, sp)

        for i in range(args.warmup):
            tc_step(i)
        torch.cuda.synchronize(dev)
        t0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        t1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        for i in range(args.steps):
            t0[i].record(stream)
            tc_step(i)
            t1[i].record(stream)
        torch.cuda.synchronize(dev)
        tc_ms = sum(a.elapsed_time(b) for a, b in zip(t0, t1)) / args.steps
        status = sg.device_status(reset=True)
        # accuracy of the last result (set (steps-1) % nsets) against the oracle on sampled rows
        tc_rrmse = None
        if rank == 0 and batch == 1 and not w.transA:
            import oracle
            dC = sets[(args.steps - 1) % nsets][2]
            rows = np.arange(0, M, max(1, M // 64))
            got = dC.view(M, ldc)[rows, :N].cpu().numpy()
            ref = oracle.sgemm(np.ascontiguousarray(case["A"][0][rows]), case["B"][0], len(rows),
                               N, K, lda=lda, ldb=ldb)
            tc_rrmse = oracle.rrmse(got, ref)
        peaks = measured_peaks()
        bf16 = peaks.get("bf16_tflops")
        tf32_peak = bf16 * TF32_PER_BF16 if bf16 else 1100.0
        tc_alg = flops / (tc_ms * 1e-3) / 1e12
        tf32_probe = tf32_probe_tflops(torch, sg, dev, stream)
        tc = {
            "value": world * tc_alg, "unit": "TFLOP/s", "ms_per_step": tc_ms,
            "kernels": tc_plan(M, N, K, batch, w.transA, w.transB, aligned, rows128, sms_dev)[0],
            "gpu_launches_per_step": tc_plan(M, N, K, batch, w.transA, w.transB, aligned,
                                             rows128, sms_dev)[1],
            "pct_of_fp32_peak_at_max_clock": None,
            "roofline": {"bound": "tensor", "achieved": 3 * tc_alg, "peak": tf32_probe,
                         "unit": "TFLOP/s", "frac": 3 * tc_alg / tf32_probe,
                         "traffic": profiled_traffic(tc_kernel_name(K), args.workload),
                         "traffic_kernel": tc_kernel_name(K),
                         "peak_source": "measured in this run: the library's TF32 tensor-pipe "
                                        "probe (sgemm_probe_tf32_mma: back-to-back "
                                        "tcgen05.mma.kind::tf32 M128 N256 K8 from shared memory, "
                                        "one CTA per SM)",
                         "note": "achieved = tensor-pipe work (3 TF32 MMAs per product) / time of "
                                 "the whole call, split kernels included",
                         "peak_bf16_derived": tf32_peak,
                         "frac_of_bf16_derived": 3 * tc_alg / tf32_peak,
                         "bf16_derived": ("measured bf16 burst x nominal TF32/BF16 ratio 1.1/2.25 "
                                          "(below what the TF32 probe reaches, so not the "
                                          "denominator)" if bf16 else "nominal dense TF32")},
            "rrmse_vs_oracle": tc_rrmse,
            "device_status": status,
        }

    # split-K on the pages' one-tile case (128 x 128 x 32768): plain vs split
    sk = None
    gemv_line = None
    if not args.no_tf32x3 and rank == 0:
        sm_, sn_, sk_ = 128, 128, 32768
        gA = torch.rand(sm_, sk_, device=dev) * 2 - 1
        gB = torch.rand(sk_, sn_, device=dev) * 2 - 1
        gC = torch.empty(sm_, sn_, device=dev)
        splits = sg.splitk_auto_splits(sm_, sn_, sk_)
        need_sk = sg.splitk_workspace_size(sm_, sn_, sk_, splits)
        wsk = torch.empty(max(need_sk, 1), dtype=torch.uint8, device=dev)

        def plain():
            sg.sgemm_f32(sm_, sn_, sk_, gA.data_ptr(), sk_, gB.data_ptr(), sn_, gC.data_ptr(), sn_,
                         0, 0, sp)

        def split():
            sg.sgemm_f32_splitk(sm_, sn_, sk_, gA.data_ptr(), sk_, gB.data_ptr(), sn_,
                                gC.data_ptr(), sn_, 0, 0, splits, wsk.data_ptr(), need_sk, sp)

        def timed(fn, reps=10):
            for _ in range(2):
                fn()
            a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(reps):
                fn()
            a1.record(stream)
            torch.cuda.synchronize(dev)
            return a0.elapsed_time(a1) / reps

        t_plain, t_split = timed(plain), timed(split)
        fl = 2.0 * sm_ * sn_ * sk_
        sk = {"shape": [sm_, sn_, sk_], "splits": splits, "sgemm_f32_ms": t_plain,
              "splitk_ms": t_split, "speedup_over_sgemm_f32": t_plain / t_split,
              "splitk_tflops": fl / (t_split * 1e-3) / 1e12,
              "note": "sgemm_f32 already splits this K over the CTAs of one 16-CTA cluster "
                      "(no workspace); sgemm_f32_splitk uses 64 chunks and a reduction pass"}
        del gA, gB, gC, wsk

        # matrix-vector shape (N = 1): bound by reading A once from HBM
        gm, gk = 8192, 8192
        vA = torch.rand(gm, gk, device=dev) * 2 - 1      # 256 MB, larger than L2
        vx = torch.rand(gk, 1, device=dev) * 2 - 1
        vy = torch.empty(gm, 1, device=dev)

        def gemv():
            sg.sgemm_f32(gm, 1, gk, vA.data_ptr(), gk, vx.data_ptr(), 1, vy.data_ptr(), 1, 0, 0, sp)

        def colsum():   # M = 1: y = x^T B with B (the same 8192 x 8192 buffer) row-major
            sg.sgemm_f32(1, gm, gk, vx.data_ptr(), gk, vA.data_ptr(), gm, vy.data_ptr(), gm, 0, 0,
                         sp)

        t_gemv = timed(gemv)
        t_colsum = timed(colsum)
        gbytes = 4.0 * (gm * gk + gk + gm)
        hbm = float(measured_peaks().get("hbm_gbs") or 6787.0)
        gemv_line = {"shape": [gm, 1, gk], "ms": t_gemv, "gbs": gbytes / (t_gemv * 1e-3) / 1e9,
                     "frac_of_hbm": gbytes / (t_gemv * 1e-3) / 1e9 / hbm,
                     "hbm_peak_gbs": hbm, "bound": "hbm",
                     "kernel": "gemv_dot_kernel (N = 1, A row-major: two rows per warp)",
                     "colsum": {"shape": [1, gm, gk], "ms": t_colsum,
                                "gbs": gbytes / (t_colsum * 1e-3) / 1e9,
                                "frac_of_hbm": gbytes / (t_colsum * 1e-3) / 1e9 / hbm,
                                "kernel": "gemv_colsum_kernel (M = 1, B row-major: K split over "
                                          "warps and a CTA cluster)"}}
        del vA, vx, vy

    # every named workload on both FP32-accuracy paths (not the timed step)
    table = None
    if not args.no_workloads and rank == 0:
        table = workload_table(torch, sg, dev, stream, sp)

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    props = torch.cuda.get_device_properties(dev)
    sms = props.multi_processor_count
    sms_for_label = sms
    peaks = measured_peaks()
    sm_max = float(peaks.get("sm_max_mhz") or clocks.get("sm_max_mhz") or SM_MAX_MHZ_DEFAULT)
    peak_max = sms * FP32_LANES_PER_SM * 2 * sm_max * 1e6 / 1e12
    per_gpu = value / world
    sm_now = clocks.get("sm_mhz")
    achieved = flops / (ms_per_step * 1e-3) / 1e12
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": args.workload, "M": M, "N": N, "K": K, "batch": batch,
                   "transA": w.transA, "transB": w.transB, "dist": w.dist,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": f"{nsets} rotating input sets of {workloads.min_bytes(M, N, K, batch) / 1e6:.0f} MB "
                         f"(> 129 MB L2 together); each step starts with its operands evicted",
                   "entry": "sgemm_f32_streamk" if batch == 1 else "sgemm_f32_strided_batched",
                   "raster_group": args.raster_group or 8,
                   "workspace_bytes": sk_need,
                   "kernels_per_step": launches,
                   "kernel": step_kernel_label(M, N, K, w.transA, w.transB, sms_dev, batch,
                                               simt_kernel_label(M, N, batch, w.transB,
                                                                 sms_for_label, K),
                                               aligned)},
        "pct_of_fp32_peak": {
            "at_max_clock": 100.0 * per_gpu / peak_max,
            "peak_tflops_at_max_clock": peak_max,
            "at_sampled_clock": (100.0 * per_gpu / (peak_max * sm_now / sm_max)) if sm_now else None,
            "sms": sms, "fp32_lanes_per_sm": FP32_LANES_PER_SM, "sm_max_mhz": sm_max,
        },
        "roofline": {
            "bound": "alu",
            "achieved": achieved,
            "peak": peak_max,
            "unit": "TFLOP/s",
            "frac": achieved / peak_max,
            "traffic": profiled_traffic(streamk_plan(M, N, K, w.transA, w.transB, sms_dev,
                                                     aligned)[2]
                                        if batch == 1 else "sgemm_simt_kernel", args.workload),
            "peak_source": f"derived: {sms} SMs x {FP32_LANES_PER_SM} FP32 lanes x 2 FLOP x "
                           f"{sm_max:.0f} MHz",
            "algorithmic_flops_per_launch": flops,
            "note": "achieved = algorithmic FLOPs / CUDA-event time of the whole call (transpose "
                    "and fix-up kernels included), so the tile kernel alone runs a little faster",
        },
        "clocks": clocks,
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": e2e_steps,
                "method": "pinned host A, B -> device, the step's call, C -> pinned host, every "
                          "step; two buffer sets on upload/compute/download streams, CUDA events"},
        "gpu_launches": args.steps * launches,
        "timing": {"mean_ms": ms_per_step, "median_ms": sorted(durs)[len(durs) // 2],
                   "min_ms": min(durs), "max_ms": max(durs),
                   "cold_l2": {"median_ms": cold[len(cold) // 2],
                               "tflops": flops / (cold[len(cold) // 2] * 1e-3) / 1e12,
                               "steps": cold_steps, "flush_bytes": 512 * 2**20,
                               "method": "512 MiB written on the stream before each call, "
                                         "outside the call's events"}},
        "wall_s": wall,
    }
    if plain_ms is not None:
        plain = flops / (plain_ms * 1e-3) / 1e12
        line["sgemm_f32"] = {
            "value": world * plain, "unit": "TFLOP/s", "ms_per_step": plain_ms,
            "pct_of_fp32_peak_at_max_clock": 100.0 * plain / peak_max,
            "kernel": simt_kernel_label(M, N, batch, w.transB, sms_for_label, K, w.transA),
            "roofline": {"bound": "alu", "achieved": plain, "peak": peak_max, "unit": "TFLOP/s",
                         "frac": plain / peak_max,
                         "traffic": profiled_traffic("sgemm_simt_tma_kernel"
                                                     if (w.transA or not w.transB) and aligned
                                                     else "sgemm_simt_kernel", args.workload)},
            "note": "the same product through plain sgemm_f32 (one kernel, no workspace)"}
    if tc is not None:
        tc["pct_of_fp32_peak_at_max_clock"] = 100.0 * tc["value"] / world / peak_max
        line["tf32x3"] = tc
    if sk is not None:
        line["splitk_one_tile"] = sk
        line["gemv"] = gemv_line
    if table is not None:
        line["workloads"] = table
    if cpu is not None:
        line["cpu_baseline"] = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample",
                                                    "per_workload") if k in cpu}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
