"""The multi-process parts of bench.py on CPU: the max-over-ranks timing
reduction as two gloo ranks, and the reference arm under two ranks (rank 0
alone measures and prints; the other rank exits 0 without work)."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(1.5 + rank, dist, "cpu")
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, start_method="spawn", join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_max_over_ranks_single_process():
    assert bench.max_over_ranks(3.25, None, "cpu") == 3.25


def _reference(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "2",
           "--warmup", "1", "--workload", "tiny", "--rows", "2", "--cpu-seconds", "1"]
    return subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)


def test_reference_arm_prints_on_rank_zero_only():
    r1 = _reference(1)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = _reference(0)
    assert r0.returncode == 0, r0.stderr[-2000:]
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
