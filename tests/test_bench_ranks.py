"""The multi-replica timing of bench.py on CPU: two gloo ranks (127.0.0.1),
each with its own step time, must both see the slowest rank's time and the
whole-job rate built from it."""
from __future__ import annotations

import multiprocessing as mp
import os
import socket
import sys

from conftest import ROOT


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        rate = bench.whole_job_rate(1000, world, ms)
        torch.distributed.barrier()
        out_q.put((rank, ms, rate))
    finally:
        torch.distributed.destroy_process_group()


def test_two_replicas_report_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    codes = [p.exitcode for p in procs]
    for p in procs:
        if p.is_alive():
            p.kill()
    assert codes == [0, 0], codes
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms, rate in got:
        assert ms == 15.0, (rank, ms)
        assert abs(rate - 2 * 1000 / 0.015) < 1e-6, (rank, rate)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.whole_job_rate(8192, 1, 2.0) == 8192 / 0.002
