"""The benchmark's multi-process path, on the CPU.

Multi-GPU here is replicas only: every rank runs its own microbatch and the
ranks exchange nothing but the timing.  These tests run that exchange with
two `gloo` ranks on the CPU, and launch the reference arm under torchrun
with two processes, where only rank 0 may print its line.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, steps, out_path):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        v = bench.job_ms_per_microbatch(times[rank], steps, world, "cpu")
        with open(f"{out_path}.{rank}", "w") as f:
            f.write(repr(v))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_over_all_microbatches(tmp_path):
    torch = pytest.importorskip("torch")
    import torch.multiprocessing as mp

    world, steps = 2, 4
    times = [40.0, 52.0]  # timed region of each rank, ms
    out = str(tmp_path / "v")
    mp.start_processes(_rank_main, args=(world, _free_port(), times, steps, out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        v = float(open(f"{out}.{r}").read())
        # 2 ranks x 4 steps = 8 microbatches in max(40, 52) ms
        assert v == pytest.approx(52.0 / 8, rel=1e-12), (r, v)
    del torch


def test_single_process_needs_no_process_group():
    pytest.importorskip("torch")
    sys.path.insert(0, ROOT)
    import bench

    assert bench.job_ms_per_microbatch(30.0, 3, 1, "cpu") == pytest.approx(10.0)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    pytest.importorskip("torch")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_global"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "ms" and rec["value"] > 0
    assert rec["config"]["parallelism"] == "replicas x2"
    assert rec["e2e"]["value"] == rec["value"] and rec["cpu_baseline"]["kind"] == "oracle"
