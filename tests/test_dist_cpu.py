"""The multi-rank path of the benchmark (one replica per rank, no data exchange) on two gloo
ranks on the CPU: the job's time is the slowest rank's, its throughput counts every rank's units."""
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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = [12.5, 20.0][rank]  # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_ms, "cpu")
    value = bench.replica_throughput(8 * 100, world, slowest)
    dist.barrier()
    out[rank] = (slowest, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_count_all_units():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    os.environ["PYTHONPATH"] = root + os.pathsep + os.environ.get("PYTHONPATH", "")
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        slowest, value = out[r]
        assert slowest == 20.0
        assert value == pytest.approx(2 * 800 / 0.020)


def test_single_rank_is_unchanged():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.replica_throughput(10, 1, 1000.0) == pytest.approx(10.0)
