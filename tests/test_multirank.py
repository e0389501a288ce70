"""The bench's multi-rank path on the CPU: world size 2 over gloo.

Every rank runs its own replica on its own requests (no exchange on the data path); the ranks
meet only to combine timings and counts.  These tests check that combination (max and sum over
ranks, whole-job throughput = units of all ranks over the slowest rank's time) with two gloo
processes, and that under torchrun the reference arm runs on rank 0 alone.
"""
import json
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def rank_worker(rank: int, world: int, port: int, out_dir: str):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, str(ROOT))
    import bench

    ranks = bench.Ranks("gloo", torch.device("cpu"))
    ranks.barrier()
    res = {
        "world": ranks.world, "rank": ranks.rank,
        "max": ranks.max(1.5 + rank),              # 2.5 on every rank
        "sum": ranks.sum(rank + 1),                # 3
        # rank r processed 10 (r + 1) units in 1 + r seconds: 30 units over the slowest 2 s
        "throughput": ranks.throughput(10 * (rank + 1), 1.0 + rank),
    }
    ranks.barrier()
    ranks.close()
    Path(out_dir, f"rank{rank}.json").write_text(json.dumps(res))


def test_ranks_combine_timings_over_two_gloo_processes(tmp_path):
    world = 2
    mp.start_processes(rank_worker, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        res = json.loads((tmp_path / f"rank{r}.json").read_text())
        assert res["world"] == world and res["rank"] == r
        assert res["max"] == 2.5
        assert res["sum"] == 3.0
        assert res["throughput"] == 15.0


def test_single_rank_needs_no_process_group(monkeypatch):
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, str(ROOT))
    import bench

    ranks = bench.Ranks("gloo", torch.device("cpu"))
    assert ranks.world == 1 and ranks.dist is None
    ranks.barrier()
    assert ranks.max(4.0) == 4.0 and ranks.sum(4.0) == 4.0
    assert ranks.throughput(12, 3.0) == 4.0
    ranks.close()


def test_reference_arm_runs_on_rank_zero_alone_under_torchrun():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           "bench.py", "--impl", "reference", "--gpus", "2", "--workload", "1", "--steps", "3",
           "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
