"""Multi-rank host logic on the CPU: gloo process groups.

The bench's multi-GPU path partitions into independent problems (every (sequence, head) chain
is independent), so N GPUs run N independent batches of the same shape with no collective on
the data path (weak scaling); the only exchange is the maximum of the ranks' timed durations.
These tests run that host logic -- per-rank inputs and the max-over-ranks reduction -- in two
CPU processes, and launch the bench's reference arm under torch.distributed.run with two ranks
(rank 0 alone runs and prints; the other exits without work).

The sequence-sharded prefill has one real exchange: the ranks' transfer pairs (B, Phi) are
all-gathered and each rank chains those of the ranks before it.  Its host logic runs here in
groups of 2 and 3 ranks, with the float64 oracle standing in for the three device steps.
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
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3", "--workload", "2"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["steps"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"


# ------------------------------------------------- sequence-sharded prefill: the host exchange

def _shard_tensors(w, cuts, r):
    """Rank r's packed shard: tokens [cuts[i][r], cuts[i][r+1]) of every sequence i."""
    M, cu = w.M, w.cu_seqlens.tolist()
    idx_t, idx_e, lens = [], [], []
    for i in range(len(cu) - 1):
        a, b = cu[i] + cuts[i][r], cu[i] + cuts[i][r + 1]
        idx_t += list(range(a, b))
        idx_e += list(range(M * a, M * b))
        lens.append(b - a)
    it, ie = torch.tensor(idx_t, dtype=torch.long), torch.tensor(idx_e, dtype=torch.long)
    cu_l = torch.tensor([0] + list(torch.tensor(lens).cumsum(0).tolist()), dtype=torch.int32)
    return dict(q=w.q[it], k=w.k[ie], v=w.v[ie], g=w.g[it], beta=w.beta[ie], cu=cu_l)


SEQPAR_LENGTHS = [90, 40, 0]


def _seqpar_cuts(world):
    # per sequence, the token boundaries of the shards of ranks 0 .. world-1 (an empty shard included)
    return {2: [[0, 37, 90], [0, 0, 40], [0, 0, 0]], 3: [[0, 20, 63, 90], [0, 40, 40, 40], [0, 0, 0, 0]]}[world]


def _seqpar_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import numpy as np
    import oracle
    import chunked_gated_deltaproduct_gb300 as pkg
    from gdp_workloads import make_custom

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        M, H, d = 2, 2, 8
        w = make_custom(SEQPAR_LENGTHS, H, d, M, seed=150, decay=0.1, init_sigma=0.5)  # every rank draws the same
        sh = _shard_tensors(w, _seqpar_cuts(world), rank)
        N = len(SEQPAR_LENGTHS)

        def transfer():  # the oracle stands in for the GPU's transfer pairs
            b = oracle.forward(sh["q"], sh["k"], sh["v"], sh["g"], sh["beta"], sh["cu"], M, w.scale)["final_state"]
            eye = torch.eye(d).expand(N, H, d, d).contiguous()
            phi = oracle.forward(sh["q"], sh["k"], torch.zeros_like(sh["v"]), sh["g"], sh["beta"], sh["cu"], M,
                                 w.scale, initial_state=eye)["final_state"]
            return torch.from_numpy(np.stack([b, phi])).float()

        def chain(s0, phi, b):  # the plain definition stands in for the GPU chain
            s = [np.zeros((N, H, d, d)) if s0 is None else s0.double().numpy()]
            for j in range(phi.shape[0]):
                s.append(s[-1] @ phi[j].double().numpy() + b[j].double().numpy())
            return torch.from_numpy(np.stack(s)).float()

        def run(s_in):
            return oracle.forward(sh["q"], sh["k"], sh["v"], sh["g"], sh["beta"], sh["cu"], M, w.scale,
                                  initial_state=s_in)

        res = pkg.sequence_parallel_steps(transfer, chain, run, w.initial_state)
        out[rank] = (res["o"].tolist(), res["final_state"].tolist())
    finally:
        dist.destroy_process_group()


import pytest  # noqa: E402


@pytest.mark.parametrize("world", [2, 3])
def test_sequence_sharded_prefill_host_exchange(world):
    """world ranks hold consecutive token shards of every sequence; the pairs exchange and the
    chaining of the ranks before each one (the library's host logic, with the oracle standing in
    for the device steps) reproduce the unsharded run: outputs in token order, the last rank's
    state = the final state."""
    import numpy as np
    import oracle
    from gdp_workloads import make_custom
    from tests._pins import rel_err

    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_seqpar_main, args=(world, port, out), nprocs=world, start_method="spawn", join=True)
    w = make_custom(SEQPAR_LENGTHS, 2, 8, 2, seed=150, decay=0.1, init_sigma=0.5)
    whole = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, 2, w.scale, initial_state=w.initial_state)
    cuts, cu = _seqpar_cuts(world), w.cu_seqlens.tolist()
    o = np.zeros_like(whole["o"])
    for r in range(world):
        o_r = np.asarray(out[r][0])
        pos = 0
        for i in range(len(SEQPAR_LENGTHS)):
            n = cuts[i][r + 1] - cuts[i][r]
            o[cu[i] + cuts[i][r]:cu[i] + cuts[i][r + 1]] = o_r[pos:pos + n]
            pos += n
    # each shard starts from the fp32 rounding of the chained state, hence the tolerance
    assert rel_err(o, whole["o"]) < 1e-6
    assert rel_err(np.asarray(out[world - 1][1]), whole["final_state"]) < 1e-6
