"""The N > 1 host path of bench.py on CPU: two gloo ranks (127.0.0.1) check
that the job time is the slowest rank's and that the whole-job µs per call
counts every replica's calls; the reference arm runs on rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    w, r, local = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    local_ms = 10.0 + 5.0 * r                  # rank 1 is the slow one
    dist.barrier()
    job_ms = bench.max_over_ranks(local_ms, "cpu")
    us = bench.us_per_call(job_ms, steps=4, world=w)
    dist.barrier()
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"world": w, "rank": r, "local": local, "job_ms": job_ms, "us": us}, f)


def test_two_rank_timing_aggregation(tmp_path):
    port = _free_port()
    tmp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    for r, d in enumerate(res):
        assert d["world"] == 2 and d["rank"] == r and d["local"] == r
        assert d["job_ms"] == 15.0                      # max over ranks, on every rank
        assert d["us"] == pytest.approx(15.0 * 1000 / (4 * 2))


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.pop(k) for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK") if k in os.environ}
    try:
        assert bench.dist_env() == (1, 0, 0)
        assert bench.us_per_call(2.0, steps=4, world=1) == 500.0
    finally:
        os.environ.update(env)


def test_reference_arm_runs_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_line_fits_its_own_clock():
    # each step times the oracle on a fixed slice of the call: the line's
    # steps x ms_per_step must fit in the process's wall time, and the
    # per-call value is marked as extrapolated from that slice
    import time
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    t0 = time.time()
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "2", "--warmup", "3", "--M", "12", "--ref-budget", "0.3"],
                       env=env, capture_output=True, text=True, timeout=600)
    wall = time.time() - t0
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["steps"] * line["ms_per_step"] / 1000 < wall
    ex = line["value_extrapolated"]
    assert 1 <= ex["from_experts"] <= ex["of_experts"]
    assert line["value"] == pytest.approx(
        ex["measured_s_per_step"] * ex["of_experts"] / ex["from_experts"] * 1e6, rel=0.01)
    assert line["metric"].endswith("M=12)")
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def test_launch_count_and_metric_follow_the_workload():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.launches_per_call(0, 6) == 0
    assert bench.launches_per_call(42, 6) == 4          # 252 routes: one front launch
    assert bench.launches_per_call(768, 6) == 5         # sort, gather, 2 GEMMs, finalise
    assert bench.launches_per_call(16384, 6) == 6       # count + scatter sort
    assert bench.metric_name(16384).endswith("M=16384)")
