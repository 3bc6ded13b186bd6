"""The benchmark's multi-rank path (one independent layer replica per rank,
barrier, max-over-ranks timing) on two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    w, r, local = bench._dist()
    assert (w, r, local) == (world, rank, rank)
    bench._barrier(w)
    # each rank reports its own "time"; every rank must see the maximum
    m = bench._max_over_ranks(w, float(10 + rank))
    out[rank] = m
    dist.destroy_process_group()


def test_two_gloo_ranks_barrier_and_max_over_ranks():
    if not dist.is_gloo_available():
        pytest.skip("gloo not available")
    world, port = 2, _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    assert dict(out) == {0: 11.0, 1: 11.0}


def test_single_rank_needs_no_process_group(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench._dist() == (1, 0, 0)
    assert bench._max_over_ranks(1, 3.5) == 3.5


def test_reference_arm_under_two_ranks_prints_once():
    """`bench.py --impl reference` launched as two ranks (gloo on the CPU):
    rank 0 times the oracle and prints the one JSON line, the other rank exits
    0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--config", "tiny_fp32_T256_E8", "--steps", "1", "--warmup", "3", "--ref-tokens", "16"]
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run(cmd, cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
