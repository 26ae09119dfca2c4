"""The multi-rank path of bench.py on the CPU (gloo, world size 2).

The decode path shards by sequence with no exchange step, so several GPUs run
independent replicas; what multi-rank code there is lives on the host: the
job time is the slowest rank's (max over ranks), and the reference arm prints
from rank 0 only.  These tests run that host logic as two gloo processes."""
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
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    results[rank] = bench.max_over_ranks(1.5 + rank, dist, torch.device("cpu"))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    # The manager's server process starts with spawn too: forking a process
    # whose threads (torch, OpenMP) are already running can deadlock.
    with mp.get_context("spawn").Manager() as mgr:
        results = mgr.dict()
        mp.spawn(_max_worker, args=(2, port, results), nprocs=2, join=True)
        assert dict(results) == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process():
    import bench
    assert bench.max_over_ranks(3.25, None, torch.device("cpu")) == 3.25


def test_reference_arm_two_ranks_prints_once():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3",
           "--workload", "tiny"]
    env = dict(os.environ, OMP_NUM_THREADS="2", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0
