"""The multi-rank bench path on CPU: two gloo ranks, each a replica with its
own bytes and time; the job reports the byte sum over the max time."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_bytes = 1000.0 * (rank + 1)
    local_seconds = 0.5 + rank
    results[rank] = bench.aggregate(local_bytes, local_seconds, world)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_sums_bytes_and_takes_max_time():
    import torch.multiprocessing as mp

    port = _free_port()
    manager = mp.get_context("spawn").Manager()
    results = manager.dict()
    mp.start_processes(_worker, args=(2, port, results), nprocs=2, join=True,
                       start_method="spawn")
    for rank in range(2):
        assert results[rank] == (3000.0, 1.5)


def test_single_rank_aggregation_is_identity():
    import bench

    assert bench.aggregate(123.0, 0.25, 1) == (123.0, 0.25)
