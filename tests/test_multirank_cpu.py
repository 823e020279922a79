"""The multi-rank (replicas) timing path of bench.py on CPU with gloo,
world size 2: every rank must end with the slowest rank's time, and the job
value must sum the replicas' FLOPs over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank, dist, "cpu")
    value = bench.whole_job_tflops(world, 2e12, ms)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_reduce_to_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    ms, value = res[0]
    assert ms == 2.0                       # the slower rank's time
    assert value == pytest.approx(2 * 2e12 / 2e-3 / 1e12)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)   # 1 TFLOP in 1 ms
