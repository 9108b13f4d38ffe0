"""The N > 1 path of bench.py on the CPU: N independent replicas (the ring
is emulated on one GPU, so there is no data-path collective); the timed
region is the slowest replica's and the value is the whole job's.  Run with
the gloo backend, world size 2, rendezvous on 127.0.0.1."""
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
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each replica times its own steps; the job is as slow as the slowest
        ms = bench.max_over_ranks(10.0 + 5.0 * rank, torch.device("cpu"))
        dist.barrier()
        out[rank] = (ms, bench.replica_throughput(1e12, 4, ms, world))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_value_gloo():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0] == out[1]
    ms, value = out[0]
    assert ms == 15.0  # the slower replica
    # 2 replicas x 4 steps x 1e12 flop in 15 ms
    assert value == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_process_needs_no_group():
    assert bench.max_over_ranks(3.5, torch.device("cpu")) == 3.5
    assert bench.replica_throughput(2e12, 10, 1000.0, 1) == pytest.approx(20.0)


def test_reference_arm_under_torchrun_two_ranks():
    """--impl reference launched like the driver launches N > 1: rank 0 times
    the oracle and prints one JSON line, the other rank exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0
    contract = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}
    assert contract <= set(rec), contract - set(rec)
    assert rec["steps"] == 1 and rec["warmup"] == 3 and rec["higher_is_better"] is True
    assert "workload" in rec["config"] and rec["e2e"]["value"] == rec["value"]
