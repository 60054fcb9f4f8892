"""The multi-rank host logic of bench.py on CPU: two gloo ranks reduce their timed totals to the
slowest rank's, and the job's value counts every rank's replica; the reference arm's non-zero
ranks exit without work or output."""
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


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 100.0 + 50.0 * rank                     # rank r timed 100 + 50 r ms
        total = bench.max_over_ranks(torch, dist, mine, "cpu")
        out.put((rank, total, bench.job_tflops(world, 1e12, 10, total)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_total_and_count_both_replicas():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == [150.0, 150.0]
    # 2 ranks x 10 steps x 1e12 FLOP in 150 ms
    assert got[0][2] == pytest.approx(2 * 10 * 1e12 / 0.150 / 1e12)
    assert got[0][2] == got[1][2]


def test_single_rank_keeps_its_own_total():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(None, None, 123.5, "cpu") == 123.5
    assert bench.job_tflops(1, 2e12, 4, 1000.0) == pytest.approx(8.0)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
