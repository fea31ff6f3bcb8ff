"""The N > 1 bench path on CPU: two gloo ranks, independent replicas.

bench.py runs one replica per GPU, times the slowest rank (max over ranks)
and reports all ranks' work over that time.  These checks run the same
helpers across two processes with the gloo backend.
"""
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local = [1.0 + rank, 5.0 - rank, 2.5]          # rank 1 is slower on the first timing
    got = bench.max_over_ranks(local, torch.device("cpu"), world)
    out[rank] = got + [bench.replica_throughput(1e12, got[0], world)]
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_sum_the_work():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        t0, t1, t2, value = res[r]
        assert (t0, t1, t2) == (2.0, 5.0, 2.5)
        # two replicas each doing 1e12 units, slowest rank 2.0 ms
        assert value == pytest.approx(2 * 1e12 / 2e-3)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3.0, 4.0], torch.device("cpu"), 1) == [3.0, 4.0]
    assert bench.replica_throughput(10.0, 1.0, 1) == pytest.approx(1e4)
