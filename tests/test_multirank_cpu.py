"""The N > 1 host logic of bench.py on CPU: two gloo ranks (127.0.0.1) whose step times
differ agree on the slowest rank's time and on the whole-job value, and the reference arm
prints from rank 0 only.  Attention shards into independent replicas with no data-path
collective, so this is the only cross-rank logic."""
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


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms_local = [2.0, 5.0][rank]
        value_local = [100.0, 40.0][rank]          # units per second at this rank's own time
        ms, value, scale = bench.whole_job(ms_local, value_local, world, torch.device("cpu"))
        q.put((rank, ms, value, scale))
    finally:
        dist.destroy_process_group()


def test_whole_job_value_uses_the_slowest_rank():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ms0, v0, s0), (r1, ms1, v1, s1) = res
    assert ms0 == ms1 == 5.0                       # max over ranks
    assert s0 == pytest.approx(2.0 / 5.0) and s1 == 1.0
    assert v0 == pytest.approx(100.0 * 0.4 * 2)    # rank 0's rate at the slowest time, x2 replicas
    assert v1 == pytest.approx(40.0 * 1.0 * 2)


def test_single_rank_needs_no_process_group():
    import bench
    ms, value, scale = bench.whole_job(3.0, 10.0, 1, torch.device("cpu"))
    assert (ms, value, scale) == (3.0, 10.0, 1.0)


def test_reference_arm_prints_on_rank_zero_only():
    import argparse
    import bench
    args = argparse.Namespace(steps=1, warmup=1)
    assert bench.run_reference(args, rank=1, world=2) is None
