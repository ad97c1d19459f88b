"""The benchmark's replica aggregation across ranks (world size 2, gloo on CPU): every rank gets
the slowest rank's time and the throughput of all ranks' bytes over it."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        local_ms = [2.0, 4.0][rank]
        ms, value = bench.aggregate_throughput(local_ms, 1_000_000_000, dist, "cpu")
        results[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_world_2():
    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
    for rank in range(2):
        ms, value = results[rank]
        assert ms == 4.0                              # the slowest rank's time
        assert abs(value - 500.0) < 1e-9              # 2 ranks x 1 GB / 4 ms


def test_single_process_aggregation():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate_throughput(2.0, 1_000_000_000)
    assert ms == 2.0 and abs(value - 500.0) < 1e-9
