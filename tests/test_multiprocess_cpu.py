"""The N > 1 host path on CPU with gloo, world size 2: the bench's barrier,
max-over-ranks timing and whole-job rate, and the reference arm launched by
torchrun (rank 0 alone runs and prints; the other rank exits 0)."""
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


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _ranks(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(world)
        ms = [3.0, 5.0][rank]                  # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, world)
        rate = bench.job_rate(4096, world, ms_max)
        out[rank] = (ms_max, rate)
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_gloo():
    port = _free_port()
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_ranks, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for rank in (0, 1):
        ms_max, rate = res[rank]
        assert ms_max == 5.0                     # the slowest rank sets the step
        assert rate == pytest.approx(2 * 4096 / 5e-3)   # all ranks' units / that time


def test_reference_arm_under_torchrun_two_ranks():
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="", MASTER_ADDR="127.0.0.1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "1", "--warmup", "0"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1                       # rank 0 only
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the same workload fields as our arm's line prints
    import bench
    from mixture_experts_ffn_softmax_gb300 import workloads as wl
    want = bench.workload_config(wl.SPECS["tiny"])
    assert {k: line["config"][k] for k in want} == want
