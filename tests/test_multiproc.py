"""The N > 1 host path of bench.py on CPU: two gloo ranks (127.0.0.1).

Each rank owns an independent batch (weak scaling, no data-path collective):
the ranks' seeds differ, the barrier returns on both, the reported time is
the maximum over ranks, and the whole-job rate counts every rank's units.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        ms = 1.0 + rank  # rank 1 is the slow one
        out[rank] = (bench.rank_seed(rank), bench.max_over_ranks(ms, world),
                     bench.whole_job_rate(1000, world, bench.max_over_ranks(ms, world)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    seeds = {res[r][0] for r in range(world)}
    assert len(seeds) == world                      # independent batches
    assert all(res[r][1] == 2.0 for r in range(world))  # max over ranks
    assert all(res[r][2] == pytest.approx(1000 * 2 / 2e-3) for r in range(world))
