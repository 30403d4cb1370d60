"""Host-side logic of the multi-rank bench path, on CPU (gloo, two ranks).

The prefill has no exchange step between GPUs (independent replicas), so the
only collectives are the barrier around the timed region and the max over
ranks of the timed milliseconds; the job value counts the work of every rank
over the slowest rank's time. The reference arm runs on rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        dist.barrier()
        ms_max = bench.max_over_ranks(ms, world)
        q.put((rank, ms_max, bench.job_value(1e12, 100, world, ms_max)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_two_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    for rank, ms_max, value in got:
        assert ms_max == 15.0  # every rank sees the slowest time
        # 2 ranks x 100 steps x 1e12 flop in 15 ms
        assert value == pytest.approx(2 * 100 * 1e12 / 0.015 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_value(2e12, 10, 1, 20.0) == pytest.approx(1000.0)


def _run_reference(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         "t5_tiny_fp32", "--steps", "1", "--warmup", "0", "--cpu-budget", "0.5", "--gpus", str(world)],
        capture_output=True, text=True, timeout=300, env=env, cwd=ROOT)


def test_reference_arm_runs_on_rank_zero_only():
    other = _run_reference(1, 2)
    assert other.returncode == 0
    assert other.stdout.strip() == ""
    first = _run_reference(0, 2)
    assert first.returncode == 0
    line = json.loads(first.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
