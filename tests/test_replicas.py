"""The bench's replica aggregation across ranks (one replica of the layer per
GPU, no data-path collective): world size 2 over gloo on the CPU.  The job's
step time is the slowest rank's, and the job's throughput counts every rank's
tokens."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, ws, port, q):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    ms = bench.replica_step_ms(10.0 + 5.0 * rank, ws)
    q.put((rank, ms, bench.replica_value(11, ws, ms)))
    dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    out = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == 15.0  # the slowest rank's step
        assert abs(value - 2 * 11 / 0.015) < 1e-6
