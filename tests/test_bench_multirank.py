"""bench.py's multi-rank aggregation with two gloo ranks on the CPU.

At expert parallelism 1 the expert path has no exchange step, so N GPUs run N
independent replicas; the only cross-rank logic is the barrier around the
timed region, the maximum of the per-rank times and the whole-job throughput.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        # rank r took (10 + r) ms for its steps and (20 - r) ms end to end
        total, e2e = bench.max_over_ranks([10.0 + rank, 20.0 - rank], world)
        value = bench.whole_job_throughput(1000.0, 5, world, total)
        dist.barrier()
        q.put((rank, total, e2e, value))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_throughput_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, total, e2e, value in got:
        assert total == 11.0 and e2e == 20.0          # the slowest rank sets the time
        assert value == pytest.approx(1000.0 * 5 * 2 / 0.011)   # all ranks' units


def test_single_process_is_identity():
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_throughput(10.0, 2, 1, 1000.0) == pytest.approx(20.0)
