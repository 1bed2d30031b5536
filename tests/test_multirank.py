"""The benchmark's multi-rank host logic on CPU with two gloo ranks: every
rank runs its own replica, rank 0 reports the slowest rank's time and the
whole-job rate; the reference arm's other ranks exit without work."""

import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [0.050, 0.080][rank]  # rank 1 is the slow replica
        ms = bench.max_over_ranks(local_ms, world)
        results[rank] = (ms, bench.whole_job_rate(ms, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_report_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        ms, rate = res[rank]
        assert ms == 0.080
        assert abs(rate - 2 * 1000.0 / 0.080) < 1e-9


def test_reference_arm_other_ranks_exit_quietly(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        rc = bench.main(["--impl", "reference", "--steps", "5", "--warmup", "3"])
    assert rc == 0 and buf.getvalue() == ""


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.whole_job_rate(0.5, 1) == 2000.0
