"""The several-GPU path runs independent replicas; its host logic (the job's
time is the slowest rank's, the job's rate counts every rank's work) is
checked here with two gloo processes on the CPU, and the reference arm's
non-zero ranks exit without work or output."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from dense_fp32_matrix_09_gb300 import replicas

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [10.0, 12.5, 11.0][rank]           # rank 1 is the slowest
        dist.barrier()
        ms = replicas.slowest(local_ms, dist, "cpu")
        q.put((rank, ms, replicas.job_tflops(2e12, ms, world)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_slowest_rank_and_job_rate(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    slow = max([10.0, 12.5, 11.0][:world])
    for rank, ms, tf in got:
        assert ms == slow                                # every rank sees the slowest time
        assert tf == pytest.approx(2e12 * world / (slow * 1e-3) / 1e12)


def test_single_process_needs_no_group():
    assert replicas.slowest(3.5) == 3.5
    assert replicas.job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)
    with pytest.raises(ValueError):
        replicas.job_tflops(1e12, 0.0, 1)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
