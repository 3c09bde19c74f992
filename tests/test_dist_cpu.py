"""The multi-rank host path of bench.py on CPU with the gloo backend (world size 2).

On this hardware the products run as independent replicas (one per GPU, no data-path collective):
the ranks only meet in a barrier around the timed region and in a MAX all-reduce of the timed
duration, and the reference arm runs on rank 0 alone.  Both are exercised here without a GPU.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, ws: int, port: int, out_dir: str) -> None:
    sys.path.insert(0, ROOT)
    import bench
    torch.distributed.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        bench._barrier(ws)
        mx = bench._max_over_ranks(1.5 * (rank + 1), ws)      # per-rank durations 1.5 and 3.0
        bench._barrier(ws)
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": mx}, f)
    finally:
        torch.distributed.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    for r in range(2):
        with open(tmp_path / f"rank{r}.json") as f:
            assert json.load(f)["max"] == 3.0                 # every rank sees the slowest rank's time


def test_reference_arm_two_ranks_prints_one_line():
    """torchrun with two ranks: rank 0 alone times the oracle and prints the only JSON line."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
