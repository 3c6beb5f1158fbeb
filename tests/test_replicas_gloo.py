"""The multi-GPU path is replicas only (the batch-min exit rule couples the
sequences of a batch, so a batch does not shard): bench.py times N
independent replicas together, takes the slowest rank's time and reports the
whole job's tokens.  Its host logic runs here as two gloo ranks on the CPU;
the reference arm (the oracle) runs on rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        slow = bench.max_over_ranks(10.0 + 5.0 * rank, "cpu")  # rank 1 is the slow one
        tput = bench.job_throughput(64, world, slow)
        out.put((rank, slow, tput))
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(60)
    assert all(p.exitcode == 0 for p in ps)
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slow, tput in got:
        assert slow == 15.0                    # every rank sees the slowest time
        assert tput == pytest.approx(2 * 64 / 15.0)  # the job's units over it


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=120, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
