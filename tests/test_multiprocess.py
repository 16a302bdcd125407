"""The N > 1 launch path on CPU: two processes over gloo.

bench.py runs one process per GPU under torch.distributed.run; with no
exchange step in the path each rank runs an independent replica, and rank 0
reports the slowest rank's time.  These tests run that plumbing with the gloo
backend on the host: the max-over-ranks reduction, and the reference arm
(the CPU oracle) launched exactly as the multi-GPU bench is, where rank 0
alone prints one JSON line and the other rank exits 0 without work.
"""

import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    v = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
    bench.barrier(world)
    out[rank] = v
    dist.destroy_process_group()


def test_max_over_ranks_gloo_two_processes():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    mp.start_processes(_max_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
