"""The multi-rank host path of bench.py on CPU: two gloo ranks, no GPU.

Every rank runs an independent replica (sequences never interact), so the only cross-rank
steps are the barrier and the max-over-ranks timing; the whole-job value is all ranks' units
over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        seconds = [2.0, 3.0][rank]          # rank 1 is the slowest
        value, slowest = bench.aggregate(1000.0, seconds, world)
        out[rank] = (value, slowest)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_rank_weak_scaling_aggregate():
    port = _free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1]
    value, slowest = out[0]
    assert slowest == pytest.approx(3.0)
    assert value == pytest.approx(2 * 1000.0 / 3.0)


def test_single_rank_is_identity():
    import bench
    assert bench.aggregate(500.0, 2.0, 1) == (250.0, 2.0)


def test_replicas_draw_disjoint_batches_of_the_same_sizes():
    import numpy as np
    import workloads
    a = workloads.workload("tiny_gdn")
    b = workloads.workload("tiny_gdn", replica=0)
    c = workloads.workload("tiny_gdn", replica=1)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.g, b.g)
    assert c.q.shape == a.q.shape and c.v.shape == a.v.shape and c.total_tokens == a.total_tokens
    assert not np.array_equal(c.q, a.q) and not np.array_equal(c.v, a.v)
