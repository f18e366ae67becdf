"""The multi-GPU contract is replicas (no data-path collective): every rank times its
own steps and the job's rate uses the slowest rank.  The host logic that combines the
ranks runs here as two gloo processes on the CPU."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, local_ms, units, out):
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms, rate = bench.whole_job_rate(local_ms[rank], units, world)
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_whole_job_rate_uses_the_slowest_rank():
    world, units = 2, 8192
    local_ms = [0.50, 0.75]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, local_ms, units, out))
             for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in res:
        assert ms == pytest.approx(0.75)                      # max over ranks, on every rank
        assert rate == pytest.approx(world * units / 0.75e-3)  # whole job: both ranks' units


def test_whole_job_rate_single_process():
    import bench
    ms, rate = bench.whole_job_rate(0.5, 8192, 1)
    assert ms == pytest.approx(0.5) and rate == pytest.approx(8192 / 0.5e-3)
