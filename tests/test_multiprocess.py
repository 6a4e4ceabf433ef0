"""The multi-process (torchrun) path of bench.py on CPU: world size 2, gloo.

The layer core has no exchange step, so N GPUs run N replicas; what is
shared is host logic -- the barrier and the max over ranks of the timed
region -- and the reference arm, which rank 0 alone runs and prints.
"""
from __future__ import annotations

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
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    dist, r, w, local = bench.dist_setup()
    assert dist is not None and r == rank and w == world and local == rank
    assert dist.get_backend() == "gloo"
    dev = torch.device("cpu")
    bench.barrier(dist, dev)
    # each rank's timed region differs; every rank gets the slowest
    mx = bench.max_over_ranks(dist, 1.0 + rank, dev)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": mx}, f)
    bench.barrier(dist, dev)
    dist.destroy_process_group()


def test_barrier_and_max_over_ranks_with_gloo(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        got = json.loads((tmp_path / f"rank{r}.json").read_text())
        assert got["max"] == 2.0


def test_reference_arm_under_torchrun_prints_once_on_rank_0():
    pytest.importorskip("numpy")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", "bench.py", "--gpus", "2",
           "--impl", "reference", "--steps", "3", "--warmup", "3", "--ref-tokens", "64"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["unit"] == "tokens/s" and d["cpu_baseline"]["kind"] == "oracle"
