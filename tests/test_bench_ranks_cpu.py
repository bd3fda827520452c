"""bench.py's multi-rank host logic on the CPU (two gloo ranks): the step time is the
slowest rank's, the whole-job value counts every rank's tokens, and the reference arm
runs on rank 0 alone (the other ranks exit 0 and print nothing)."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank,
                            world_size=world)
    try:
        local_ms = [0.70, 0.75][rank]           # rank 1 is the slower one
        ms = bench.max_over_ranks(local_ms, world, "cpu")
        assert ms == 0.75
        assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0   # one rank: its own time
    finally:
        dist.destroy_process_group()


def test_step_time_is_the_slowest_ranks():
    import torch.multiprocessing as mp
    mp.spawn(_rank_main, args=(2, _free_port()), nprocs=2, join=True)


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-500:]
    assert out.stdout.strip() == ""
