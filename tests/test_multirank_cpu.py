"""The replicas-only multi-process path on CPU: two gloo ranks.

The path has no exchange step; ranks only meet at the timing barrier and the
max over ranks of the timed region. These tests run that code with two
processes on the host (no GPU), and run the bench's reference arm under
torchrun, where rank 0 alone times and prints and rank 1 exits without work.
"""

from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    class A:  # the fields dist_setup reads
        pass

    w, r, _ = bench.dist_setup(A())
    assert (w, r) == (world, rank)
    bench.barrier(w)
    # each rank's timed region differs; every rank must report the slowest
    t = bench.max_over_ranks(1.5 + rank, w, torch.device("cpu"))
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": t}, f)
    dist.destroy_process_group()


def test_barrier_and_max_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True, start_method="spawn")
    got = [json.load(open(tmp_path / f"rank{r}.json"))["max"] for r in range(2)]
    assert got == [2.5, 2.5]


@pytest.mark.timeout(300)
def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--workload", "cpu_small", "--steps", "2", "--warmup", "1",
           "--reference-budget", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=280, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
