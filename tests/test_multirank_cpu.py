"""The N > 1 bench path on CPU: two gloo ranks (spawned processes), each a
replica with its own time; every rank must see the slowest rank's time and
the whole-job value must sum both ranks' bytes over that time."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        ms = bench.max_over_ranks(local_ms, dist, "cpu")
        value = bench.whole_job_gbs(w, 1_000_000_000, 100, ms)
        out[rank] = (w, r, ms, value)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_max_time_and_whole_job_value():
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        w, rr, ms, value = out[r]
        assert (w, rr) == (world, r)
        assert ms == 15.0                      # the slowest rank's time, on every rank
        assert value == pytest.approx(2 * 1e9 * 100 / 15e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_gbs(1, 2e9, 10, 1000.0) == pytest.approx(20.0)
