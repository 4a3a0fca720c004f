"""The multi-rank path of bench.py on CPU: replicas only, no data-path
collective; the timing is the max over ranks (gloo, world size 2)."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_dist_env(monkeypatch):
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (1, 2, 1)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k)
    assert bench.dist_env() == (0, 1, 0)


def test_job_tops_counts_every_rank():
    import bench

    assert bench.job_tops(1, 2e12, 1000.0) == pytest.approx(2.0)
    assert bench.job_tops(2, 2e12, 1000.0) == pytest.approx(4.0)
    assert bench.slowest_rank([3.0, 4.0], None, None) == [3.0, 4.0]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    import torch

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    got = bench.slowest_rank([1.0 + rank, 10.0 - rank], dist, torch.device("cpu"))
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump(got, f)
    dist.barrier()
    dist.destroy_process_group()


def test_slowest_rank_over_gloo(tmp_path):
    import torch.multiprocessing as mp

    port = free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        assert json.load(open(tmp_path / f"rank{r}.json")) == [2.0, 10.0]


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched as the driver launches it for N = 2:
    rank 0 prints one JSON line, rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
    # the launcher's OMP_NUM_THREADS=1 does not starve the only working rank
    assert d["cpu_baseline"]["cores"] == len(os.sched_getaffinity(0))
