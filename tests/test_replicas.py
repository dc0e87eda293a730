"""The benchmark's multi-process path on CPU: two gloo ranks running the helpers
the GPU job uses (the job's time is its slowest rank's, throughput counts every
replica, each replica decodes its own sequences), and the reference arm, which
only rank 0 runs."""

import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank, dist, "cpu")  # rank 1 is the slower replica
    q.put((rank, ms, bench.job_tok_s(ms, world, 1), bench.job_tok_s(ms, world, 8), bench.replica_seed(rank)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_are_timed_by_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(q.get(timeout=180) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert [r[1] for r in res] == [2.0, 2.0]
    assert res[0][2] == pytest.approx(1000.0)  # 2 replicas x 1 token per 2 ms
    assert res[0][3] == pytest.approx(8000.0)  # 8 sequences per replica
    assert res[0][4] != res[1][4]


def test_one_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tok_s(2.0, 1, 1) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "2",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
