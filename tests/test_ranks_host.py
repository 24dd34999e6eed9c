"""Host logic of the multi-process benchmark path on CPU: two gloo ranks reduce
their timings to the maximum and compute the whole-job rate; under a launcher
only rank 0 prints the reference arm's line.  No GPU."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 0 is faster on the first timing, slower on the second
        mine = [1.0 + rank, 5.0 - rank, 0.25 * (rank + 1)]
        got = bench.max_over_ranks(mine, world)
        out.put((rank, got, bench.whole_job_rate(world, 100, got[0])))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p_ in procs:
        p_.start()
    res = dict((r, (g, v)) for r, g, v in (q.get(timeout=120) for _ in procs))
    for p_ in procs:
        p_.join(timeout=120)
        assert p_.exitcode == 0
    for r in range(2):
        got, rate = res[r]
        assert got == [2.0, 5.0, 0.5]          # max over ranks of each timing
        assert rate == pytest.approx(2 * 100 / 2.0)


def test_single_process_keeps_its_timings():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], 1) == [1.5, 2.5]
    assert bench.whole_job_rate(1, 30, 1.5) == pytest.approx(20.0)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
