"""The N > 1 path of bench.py on CPU: two gloo ranks (replicas only, no data-path
collective).  The step time reported is the slowest rank's, every rank agrees on it, the
whole-job value counts every replica's bytes, and the reference arm runs on rank 0 only."""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [1.25, 2.5][rank]
        results[rank] = bench.max_over_ranks(dist, torch, local_ms, "cpu")
        dist.barrier()
        # the reference arm: rank 0 alone prints; other ranks return without work
        buf = io.StringIO()
        if rank != 0:
            with redirect_stdout(buf):
                bench.run_reference(type("A", (), {"workload": "tiny", "layers": 0, "cpu_budget": 0.1,
                                                    "steps": 1, "warmup": 3})())
            results[10 + rank] = buf.getvalue()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_step():
    port = _free_port()
    with mp.Manager() as mgr:
        results = mgr.dict()
        mp.start_processes(_rank_main, args=(2, port, results), nprocs=2, start_method="spawn")
        assert results[0] == pytest.approx(2.5) and results[1] == pytest.approx(2.5)
        assert results[11] == ""


def test_whole_job_value_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbs(10**9, 1, 2.0)
    assert one == pytest.approx(500.0)
    assert bench.whole_job_gbs(10**9, 4, 2.0) == pytest.approx(4 * one)
