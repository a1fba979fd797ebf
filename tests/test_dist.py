"""The multi-process (N > 1) paths of bench.py on the CPU, world size 2, over
gloo: the barrier and the max-over-ranks reduction that the timed region
uses, and the reference arm under torch.distributed.run, where rank 0 alone
runs the oracle and prints one JSON line and the other rank exits 0 without
work. No GPU is involved (the bench's own arm runs replicas on GPUs; there is
no data-path collective to test)."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.skipif(torch.cuda.is_available(), reason="CPU (gloo) test of the multi-process host logic")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(dist)
        mx = bench.max_over_ranks(dist, 1.5 + rank)  # rank r reports 1.5 + r
        q.put((rank, mx))
    finally:
        dist.destroy_process_group()


def test_barrier_and_max_over_ranks_gloo():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.start_processes(_worker, args=(world, port, q), nprocs=world, join=True, start_method="spawn")
    got = dict(q.get(timeout=60) for _ in range(world))
    assert got == {0: 2.5, 1: 2.5}  # every rank sees the slowest rank's time


def test_reference_arm_two_ranks_rank0_reports():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", PYTHONUNBUFFERED="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--config", "tiny_f32", "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
