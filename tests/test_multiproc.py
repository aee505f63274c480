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
