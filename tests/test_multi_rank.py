"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

The hot path has no exchange step, so N GPUs run N independent replicas of the
step; the only cross-rank work is taking the slowest rank's time and turning it
into a whole-job throughput.  Each rank here reports a different time; both must
get the maximum, and the throughput must count every rank's units.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")
    value = bench.job_throughput(1000.0, world, ms)
    q.put((rank, ms, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in got:
        assert ms == pytest.approx(15.0)
        # 2 ranks x 1000 units in 15 ms
        assert value == pytest.approx(2000.0 / 15e-3)


def test_single_process_is_its_own_maximum():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, "cpu") == 3.25
    assert bench.job_throughput(8192, 1, 2.0) == pytest.approx(8192 / 2e-3)
