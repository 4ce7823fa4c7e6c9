"""The multi-rank logic of bench.py on CPU (gloo, two ranks on 127.0.0.1):
the max-over-ranks timing, the whole-job rate from it, the barrier, and the
reference arm's rule that only rank 0 works under torchrun."""

import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [12.5, 30.25][rank]                       # the ranks' own timed regions
        ms_max = bench.reduce_max(ms, world)
        dist.barrier()
        rate = bench.whole_job_rate(100.0, 10, ms_max, world)
        q.put((rank, ms_max, rate))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_time_and_whole_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms_max, rate in got:
        assert ms_max == 30.25                         # both ranks see the slowest rank
        assert rate == pytest.approx(2 * 100.0 * 10 / 30.25e-3)


def test_whole_job_rate_single_rank():
    import bench
    assert bench.whole_job_rate(5.0, 4, 2.0, 1) == pytest.approx(5.0 * 4 / 2.0e-3)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""
