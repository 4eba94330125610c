"""The multi-GPU bench path runs independent replicas: no data-path collective, a barrier
around the timed region, and the job's rate taken over its slowest rank.  The aggregation
helpers are exercised here on two gloo ranks on the CPU (the layer itself has no exchange
step on one node)."""
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    dist.barrier()
    # rank r took 100 * (r + 1) ms for 1000 tokens and measured (r + 1) * 1000 tokens/s end to end
    value, ms = bench.job_throughput(1000.0, 100.0 * (rank + 1), dist, device="cpu")
    e2e = bench.job_rate_min(1000.0 * (rank + 1), dist, device="cpu")
    dist.barrier()
    out[rank] = (value, ms, e2e)
    dist.destroy_process_group()


def test_two_replicas_aggregate_over_the_slowest_rank():
    ws = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:  # no fork of this (multi-threaded) process
        out = m.dict()
        mp.spawn(_rank_main, args=(ws, port, out), nprocs=ws, join=True)
        res = dict(out)
    for r in range(ws):
        value, ms, e2e = res[r]
        assert ms == 200.0                    # the slowest rank sets the job time
        assert value == pytest.approx(2 * 1000.0 / 0.2)  # tokens of all ranks / job time
        assert e2e == pytest.approx(2 * 1000.0)           # slowest rank's rate x ranks


def test_single_rank_is_plain_rate():
    sys.path.insert(0, ROOT)
    import bench
    value, ms = bench.job_throughput(500.0, 250.0)
    assert ms == 250.0 and value == pytest.approx(2000.0)
    assert bench.job_rate_min(123.0) == 123.0
