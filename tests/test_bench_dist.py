"""The multi-rank side of bench.py on CPU: two gloo ranks (no GPU), max-over-ranks timing and
summed units, and the reference arm running on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (r + 1) seconds for 10 units: job time is the slowest rank, units add up
        t_max, rate = bench.aggregate_over_ranks(float(rank + 1), 10.0, world)
        out[rank] = (t_max, rate)
        args = type("A", (), {"steps": 1, "warmup": 0, "workload": "mixtral_bf16"})()
        if rank != 0:
            # the reference arm does no work on ranks other than 0
            assert bench.bench_reference(args, rank, world) is None
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_total_units():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()   # no fork: other tests may have started threads
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        t_max, rate = out[rank]
        assert t_max == 2.0                       # the slower rank decides
        assert rate == pytest.approx(20.0 / 2.0)  # both ranks' units over the job time


def test_single_rank_aggregate_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate_over_ranks(0.5, 10.0, 1) == (0.5, 20.0)
