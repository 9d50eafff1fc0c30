"""The multi-rank logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

Each rank runs an independent replica (no data-path collective); the only
collectives are the timing barrier and the max over ranks, which these tests
exercise with per-rank timings."""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    assert bench.dist_env() == (rank, rank, world)
    bench.barrier(world)
    local_ms = 10.0 * (rank + 1)                     # rank 1 is the slow one
    ms_per_step, value = bench.aggregate(local_ms, steps=5, step_bytes=1_000_000, world=world)
    results[rank] = (ms_per_step, value, bench.max_over_ranks(float(rank), world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_rank_and_count_all_bytes():
    world = 2
    port = _free_port()
    with mp.Manager() as manager:
        results = manager.dict()
        mp.spawn(_worker, args=(world, port, results), nprocs=world, join=True)
        res = dict(results)
    for rank in range(world):
        ms_per_step, value, max_rank = res[rank]
        assert ms_per_step == pytest.approx(20.0 / 5)              # slowest rank: 20 ms over 5 steps
        assert value == pytest.approx(world * 1_000_000 / 4e-3 / 1e9)
        assert max_rank == world - 1


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.5, 1) == 3.5
    ms, value = bench.aggregate(8.0, steps=4, step_bytes=2_000_000, world=1)
    assert ms == 2.0 and value == pytest.approx(2_000_000 / 2e-3 / 1e9)
