"""The multi-GPU path of bench.py is replicas only (the layer does not shard on one GPU's
worth of experts): each rank runs the whole layer on its own inputs, the job's time is
the slowest rank's, and the job's rate counts every rank's tokens. These CPU tests run the
cross-rank pieces on two gloo ranks, and the reference arm's rank rule."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_time_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: 15.0, 1: 15.0}


def test_whole_job_rate_counts_every_replica():
    assert bench.max_over_ranks(7.5, "cpu") == 7.5          # no process group: itself
    one = bench.whole_job_rate(1, 8192, 5, 100.0)
    assert one == 8192 * 5 / 0.1
    assert bench.whole_job_rate(2, 8192, 5, 100.0) == 2 * one


def test_reference_arm_runs_on_rank_0_only():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
