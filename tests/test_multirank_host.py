"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks.

bench.py runs independent replicas (the GEMM needs no exchange): each rank
times its own steps, the slowest rank's time is taken (MAX all-reduce) and the
value is the work of all ranks over that time.  The reference arm runs on
rank 0 only; other ranks exit without work.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = [120.0, 150.0][rank]
        m = bench.reduce_max_over_ranks(per_rank_ms)
        v = bench.weak_scaling_tflops(2e12, 10, m, world)
        out.put((rank, m, v))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, v in got:
        assert m == 150.0                       # max over ranks
        assert abs(v - 2 * 2e12 * 10 / 0.150 / 1e12) < 1e-9   # both ranks' work over that time


def test_single_process_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max_over_ranks(42.0) == 42.0
    assert bench.weak_scaling_tflops(1e12, 4, 2000.0, 1) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), dict(workload=bench.WORKLOAD, steps=1, warmup=0))()
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(args) == 0
    assert buf.getvalue() == ""
