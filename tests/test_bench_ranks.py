"""The benchmark's multi-rank path on CPU (gloo, world size 2): the job time is
the slowest rank's, the rate counts every rank's bytes, and the reference arm
under torch.distributed.run prints one line from rank 0 only."""
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


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(1.0 + rank, world, "cpu")
        v = bench.job_rate(t, 1_000_000, world)
        with open(f"{out_path}.{rank}", "w") as f:
            json.dump({"t": t, "v": v}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo():
    import torch.multiprocessing as mp
    port = _free_port()
    out_dir = os.path.join(ROOT, "_build")  # git-ignored build folder of the repo
    os.makedirs(out_dir, exist_ok=True)
    out = os.path.join(out_dir, f"ranks_{os.getpid()}")
    mp.spawn(_rank_main, args=(2, port, out), nprocs=2, join=True)
    try:
        for r in range(2):
            with open(f"{out}.{r}") as f:
                d = json.load(f)
            assert d["t"] == 2.0  # the slower rank's 2 ms, seen by both
            assert abs(d["v"] - 2 * 1_000_000 / 2e-3 / 1e9) < 1e-12
    finally:
        for r in range(2):
            if os.path.exists(f"{out}.{r}"):
                os.remove(f"{out}.{r}")


def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"
