"""The benchmark's multi-rank host logic on CPU: two gloo ranks (the GPU run
uses the same calls over NCCL, one replica per GPU, no data-path exchange)."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower replica
        job_ms = bench.max_over_ranks(ms, world, device="cpu")
        dist.barrier()
        q.put((rank, job_ms, bench.job_rate(1000.0, world, job_ms / 4)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    import socket
    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, job_ms, rate in got:
        assert job_ms == 15.0                       # the max over ranks, on every rank
        assert rate == pytest.approx(2 * 1000.0 / (15.0 / 4 * 1e-3))  # both replicas' work / job time


def test_reference_arm_on_a_nonzero_rank_does_no_work():
    """Under torchrun only rank 0 runs the oracle and prints; rank 1 exits 0 silently."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
