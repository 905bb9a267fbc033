"""The N > 1 host path of bench.py on CPU: two gloo ranks (one process per
GPU when run on GPUs; replicas, no data-path collective)."""
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


def test_job_time_is_the_slowest_rank_gloo():
    import torch.multiprocessing as mp

    import multirank_worker

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=multirank_worker.timing_rank, args=(r, 2, port, 10.0 + 5.0 * r, q))
             for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r for r, _, _ in out] == [0, 1]
    for _, job_ms, tflops in out:
        assert job_ms == 15.0                                   # max over ranks
        assert tflops == pytest.approx(2 * 2.0e9 * 10 / 15e-3 / 1e12)  # both ranks' work / the job's time


def test_single_process_time_is_its_own():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.5, None) == 7.5
    assert bench.job_throughput(1, 1.0e12, 4, 1000.0) == pytest.approx(4.0)


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the reference arm runs on rank 0 alone; other ranks
    exit 0 without work or output."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_rank_zero_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="2", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "square256", "--steps", "2", "--warmup", "3", "--reference-budget-s", "2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
