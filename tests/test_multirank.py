"""The N > 1 bench path on CPU: two gloo ranks reduce their step times to the max and
report the whole-job throughput (independent replicas, no data-path collective)."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [2.0, 3.5][rank]
    ms = bench.reduce_step_time(ms_local, world, device="cpu")
    out[rank] = (ms, bench.job_throughput(bench.OPS_STEP, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
    import bench
    want = world * bench.OPS_STEP / 3.5e-3 / 1e12
    for r in range(world):
        ms, value = out[r]
        assert ms == 3.5
        assert value == pytest.approx(want)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_step_time(1.25, 1) == 1.25
    assert bench.job_throughput(2e12, 1000.0, 1) == pytest.approx(2.0)
