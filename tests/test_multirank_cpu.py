"""The multi-rank host logic of bench.py on CPU: two gloo ranks.

bench.py runs one independent replica per rank (the layer has no data-path
exchange); what ranks share is the barrier around the timed region, the
maximum of the ranks' step times, the whole-job value computed from it, and
the rule that only rank 0 runs and prints the reference arm.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, ws: int, port: int, q) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(ws), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    dist.init_process_group("gloo", rank=rank, world_size=ws, init_method=f"tcp://127.0.0.1:{port}")
    try:
        import bench
        assert bench.dist_env() == (ws, rank, rank)
        bench.barrier(ws)
        ms = bench.max_over_ranks(1.5 + rank, ws)  # rank r took 1.5 + r ms
        value = bench.job_value(ws, 4096, ms)
        # the reference arm: ranks other than 0 leave at once and print nothing
        printed = ""
        if rank != 0:
            buf = io.StringIO()
            with redirect_stdout(buf):
                bench.run_reference(bench_args())
            printed = buf.getvalue()
        bench.barrier(ws)
        q.put((rank, ms, value, printed))
    finally:
        dist.destroy_process_group()


def bench_args():
    import argparse
    return argparse.Namespace(gpus=2, steps=1, warmup=0, workload="tiny", impl="reference", no_extra=True,
                              no_cpu=True, cpu_budget=1.0)


def test_two_gloo_ranks_share_the_slowest_time_and_only_rank0_reports():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
            pytest.fail("a rank did not finish")
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(ws))
    for rank, ms, value, printed in res:
        assert ms == pytest.approx(2.5)                       # the slower rank's time, on every rank
        assert value == pytest.approx(2 * 4096 / 2.5e-3)      # tokens of both ranks / that time
        if rank != 0:
            assert printed == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.job_value(1, 4096, 2.0) == pytest.approx(4096 / 2e-3)
    bench.barrier(1)
