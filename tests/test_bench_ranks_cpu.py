"""bench.py on the CPU.  Its multi-rank host logic, as two gloo ranks: the step time is
the slowest rank's, and the reference arm runs on rank 0 alone (the other ranks exit 0
and print nothing).  And the reference arm's JSON line at N = 1."""
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
                          "--steps", "1", "--warmup", "0", "--ref-tokens", "512"], cwd=ROOT,
                         env=env,
                         capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-500:]
    assert out.stdout.strip() == ""


def test_reference_arm_line_keeps_the_contract():
    """At N = 1 the reference arm (the oracle on the host cores) prints one JSON line with
    the contract's keys, its own cpu_baseline and an e2e that moves no bytes."""
    import json
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "3", "--ref-tokens", "512"], cwd=ROOT, env=env,
                         capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-500:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1, out.stdout[-500:]
    r = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in r, key
    assert r["impl"] == "reference" and r["n_gpus"] == 1 and r["steps"] == 1
    assert r["warmup"] >= 3 and r["value"] > 0 and r["higher_is_better"] is True
    assert r["config"]["workload"].startswith("l27b_bf16")
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == r["value"] and cb["cores"] >= 1
    assert cb["unit"] == r["unit"] and cb["sample"]
    assert r["e2e"] == {"value": r["value"], "unit": r["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
