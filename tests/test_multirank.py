"""The bench's multi-GPU path on the CPU: world_size-2 process groups on gloo.

The path partitions into independent problems (every (sequence, head) chain is independent),
so N GPUs run N independent batches of the same shape with no collective on the data path
(weak scaling); the only exchange is the maximum of the ranks' timed durations.  These tests
run that host logic -- per-rank inputs and the max-over-ranks reduction -- in two CPU
processes, and launch the bench's reference arm under torch.distributed.run with two ranks
(rank 0 alone runs and prints; the other exits without work).
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


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    from gdp_workloads import make_workload

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = make_workload(2, seed=bench.rank_seed(2, rank))
        sig = torch.tensor([float(w.q.float().sum()), float(w.T), float(w.H)], dtype=torch.float64)
        sigs = [torch.zeros(3, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(sigs, sig)
        mx = bench.max_over_ranks(0.25 + rank, dist, torch.device("cpu"))
        out[rank] = (tuple(float(x) for s_ in sigs for x in s_), mx)
    finally:
        dist.destroy_process_group()


def test_replicas_draw_independent_inputs_and_reduce_the_max():
    world, port = 2, _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    (sigs0, mx0), (sigs1, mx1) = out[0], out[1]
    assert sigs0 == sigs1  # every rank saw the same gathered signatures
    q0, T0, H0, q1, T1, H1 = sigs0
    assert (T0, H0) == (T1, H1) and q0 != q1  # same shape, independent draws
    assert mx0 == mx1 == 1.25  # the slowest rank's duration


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
