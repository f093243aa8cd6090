"""The multi-GPU path is independent replicas (every (batch, head, query
tile) is independent; no collective on the data path).  Its only exchange is
the max-over-ranks of the timing, checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms, value = bench.replica_throughput(times[rank], 1e12, world, torch.device("cpu"))
        out[rank] = (ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_replica_throughput_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        times = [2.0, 5.0]  # ms: rank 1 is the slow one
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(2):
            ms, value = out[r]
            assert ms == pytest.approx(5.0)
            # two ranks x 1 TFLOP in 5 ms = 400 TFLOPS, on every rank
            assert value == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_replica_throughput_single_rank():
    import bench
    ms, value = bench.replica_throughput(4.0, 2e12, 1, torch.device("cpu"))
    assert ms == 4.0 and value == pytest.approx(500.0)
