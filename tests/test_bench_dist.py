"""The benchmark's multi-process path (replicas, max-over-ranks timing, whole-job throughput) on
CPU with the gloo backend and two ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r processed 100 tokens in (1 + r) seconds: the job took max = world seconds
        value, tmax = bench.aggregate(100.0, 1.0 + rank, world)
        out[rank] = (value, tmax)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        value, tmax = res[r]
        assert tmax == pytest.approx(2.0)
        assert value == pytest.approx(100.0 * world / 2.0)


def test_single_rank_aggregation():
    import bench
    assert bench.aggregate(50.0, 0.5, 1) == (100.0, 0.5)
    c = bench.layer_counters(__import__("synth").CONFIGS["decode"], 64, 126, 0)
    assert c["flops"] == 64 * 8 * 6 * 2048 * 768
    assert c["gemm1_swiglu"] > 126 * 2 * 768 * 2048 * 9 // 16
