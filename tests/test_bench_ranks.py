"""Host-side logic of the multi-rank bench (replicas, one process per GPU):
the whole-job times are the slowest rank's, the rate counts every rank's
units.  Run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r reports times (r + 1) ms and 10 (r + 1) s
    got = bench.rank_max([rank + 1.0, 10.0 * (rank + 1)], "cpu")
    out[rank] = got
    dist.destroy_process_group()


def test_rank_max_takes_the_slowest_rank():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == [2.0, 20.0]
    assert res[1] == [2.0, 20.0]


def test_rank_max_without_process_group():
    import bench
    assert bench.rank_max([3.0, 4.5], "cpu") == [3.0, 4.5]


@pytest.mark.parametrize("world,units,secs,want", [(1, 20, 2.0, 10.0), (2, 20, 2.0, 20.0),
                                                   (8, 5, 0.5, 80.0)])
def test_whole_job_rate(world, units, secs, want):
    import bench
    assert bench.whole_job_rate(world, units, secs) == pytest.approx(want)
