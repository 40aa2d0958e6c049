"""Replica runs (bench.py under torchrun): each rank decodes its own batch
and the job time is the slowest rank's. Checked with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method="env://")
    import bench
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    # rank r pretends its timed region took 10 * (r + 1) ms
    results[rank] = bench.max_over_ranks(10.0 * (rank + 1), world, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(results) == {0: 20.0, 1: 20.0}


def test_replica_workloads_differ_by_rank():
    """Weak scaling: each rank draws its own batch (seed = rank)."""
    from workloads import make_workload
    a = make_workload(B=1, Hq=2, Hkv=2, d=64, t=64, steps=2, N=8, seed=0)
    b = make_workload(B=1, Hq=2, Hkv=2, d=64, t=64, steps=2, N=8, seed=1)
    assert not (a.K == b.K).all()


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
