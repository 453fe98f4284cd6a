"""The benchmark's multi-rank path (independent replicas, weak scaling): with
two gloo ranks on CPU the job time is the slowest rank's and the throughput
counts both ranks' work."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms_local = 10.0 if rank == 0 else 12.5
    ms, value = bench.aggregate_step_time(ms_local, 5e12, world, dist, None)
    dist.barrier()
    out[rank] = (ms, value)
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_slowest_rank():
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        ms, value = res[rank]
        assert ms == pytest.approx(12.5)
        assert value == pytest.approx(2 * 5e12 / 12.5e-3 / 1e12)


def test_single_rank_aggregation():
    import bench
    ms, value = bench.aggregate_step_time(8.0, 4e12, 1)
    assert ms == 8.0 and value == pytest.approx(4e12 / 8e-3 / 1e12)
