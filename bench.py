"""Bench: real tokens/s of the GDP varlen prefill on one GB300 (device-timed),
with the roofline fractions, an end-to-end leg through host buffers, and the
float64 CPU oracle as the reported CPU baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 4] [--impl gdp|reference]

The headline workload is the largest single-GPU configuration: one sequence of
65536 tokens (131072 expanded rows), H=32, d=128, M=2, initial state, final
state and per-chunk states.  A step is one full gdp_prefill_varlen call over
that batch, inputs resident in HBM.  Between timed steps a 256 MiB buffer is
written to flush the 129 MB L2.  The timed steps are plain gdp_prefill_varlen
calls, each bracketed by CUDA events on the launching stream; a second pass of
the same steps through gdp_prefill_varlen_profiled, whose events sit between
the stages (so each stage runs alone), gives the per-stage durations.

Reported beside the headline (key per_workload): the other benchmark
configurations -- the four-sequence varlen batch (1421 tokens, H8, M2, chunk
states), the 8 x 4096 batch (H16, M3, in-kernel L2 norm) and the serving step
(64 log-uniform sequences, H16, M4, state cache in place, prebuilt descriptors)
timed as a CUDA-graph replay.  Also reported: the decode step (key
decode_step) and the backward pass of the headline workload (key backward).
Under torchrun every rank runs its own independent batch of the same shape
(weak scaling, no collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from gdp_workloads import make_custom, WORKLOADS, make_workload  # noqa: E402

METRIC = "GDP prefill real tokens/s on 1 GB300 (device-timed) and % of roofline"
UNIT = "tokens/s"
HEADLINE_WORKLOAD = 4
PER_WORKLOAD = (2, 3, 5)
FALLBACK_HBM_GBS = 6800.0
# DRAM traffic of a stage per call, from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum summed over the stage's kernels, scaled to the full call where the
# capture ran a reduced shape), keyed by (stage, workload id); each entry names the source
# files of the stage's kernels and the sha256 of those files when the capture was taken, and is
# reported as null once they change.
NCU_TRAFFIC = {
    # the 65536-token sequence: its segmented stage runs 16 scan launches of 128 expanded chunks x
    # 32 heads and 15 WY segments of 4096 tiles beside them.  Captured on the 12288-token cut of
    # the same shape (profile_case w4): one middle-segment scan launch, 506071808 + 145328896 B,
    # and one WY segment, 171891200 + 443047168 B (both launches cover exactly one full segment).
    ("gdp_scan_kernel x16 (segmented, WY segments 2.. beside it)", 4): {
        "sources": ["gdp_scan_body.cuh", "gdp_scan.cu", "gdp_wy_body.cuh", "gdp_wy.cu", "gdp_sm100.cuh",
                    "gdp_internal.cuh"],
        "sha": "71d1476e59c6c77a",
        "bytes_per_call": 16 * (506071808 + 145328896) + 15 * (171891200 + 443047168),
    },
}


def alg_bytes(w) -> int:
    """Algorithmic bytes of one call: inputs read once, outputs written once
    (q, o bf16; M x (k, v) bf16; g fp32; M x beta fp32 per token-head) plus the
    fp32 states read and written and the requested chunk states."""
    d, M, H = w.d, w.M, w.H
    b_tok = 2 * d * (1 + 2 * M + 1) + 4 + 4 * M
    total = b_tok * w.T * H
    st = d * d * 4
    if w.initial_state is not None:
        total += w.N * H * st
    if w.state is not None:
        live = int((w.state_indices >= 0).sum())
        total += 2 * live * H * st  # slot read + slot write
    elif w.output_final_state:
        total += w.N * H * st
    if w.return_chunk_states:
        total += w.NT * H * st
    return int(total)


def alg_flops(w) -> float:
    """Dense-tile flops per expanded chunk (r rows, q = r/M readout rows)."""
    d, M = w.d, w.M
    f = 0.0
    for L in w.lengths:
        rows = L * M
        for c in range(0, rows, 64):
            r = min(64, rows - c)
            q = r / M
            f += 2 * r * r * d + r ** 3 / 3 + 4 * r * r * d + 4 * r * d * d + 2 * q * d * d + 4 * q * r * d
    return f * w.H


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            j = json.load(fh)
        return float(j.get("hbm_gbs", FALLBACK_HBM_GBS)), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, folder: str | None = None):
        self.index, self.proc, self.path = index, None, None
        self.folder = folder or tempfile.gettempdir()  # where the raw samples go (--clocks-dir)

    def __enter__(self):
        try:
            os.makedirs(self.folder, exist_ok=True)
            self.path = os.path.join(self.folder, f"clocks_bench_{os.getpid()}.csv")
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def sources_sha(files) -> str:
    """sha256 (16 hex digits) of the given files under the package's csrc/ folder."""
    h = hashlib.sha256()
    for name in files:
        p = os.path.join(ROOT, "chunked_gated_deltaproduct_gb300", "csrc", name)
        if not os.path.exists(p):
            return ""
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


# ------------------------------------------------------------------------- the oracle's sample

def oracle_sample(w, frac: float) -> dict:
    """Every head, each sequence cut to its first ceil(frac * L) tokens: the bounded sample of
    the workload that the CPU baseline and the reference arm time (all heads, so that the
    oracle's parallel loop over (sequence, head, V-row block) has the workload's own width)."""
    lens = [min(L, max(1, int(math.ceil(L * frac)))) if L else 0 for L in w.lengths]
    cu = w.cu_seqlens.tolist()
    parts = [torch.arange(cu[i], cu[i] + lens[i]) for i in range(w.N)]
    tok = torch.cat(parts) if parts else torch.arange(0)
    rows = (tok[:, None] * w.M + torch.arange(w.M)[None]).reshape(-1)
    sub_cu = [0]
    for L in lens:
        sub_cu.append(sub_cu[-1] + L)
    return {"q": w.q[tok], "k": w.k[rows], "v": w.v[rows], "g": None if w.g is None else w.g[tok],
            "beta": None if w.beta is None else w.beta[rows], "cu": sub_cu, "T": int(tok.numel())}


def _oracle_run(oracle, w, s, threads):
    oracle.forward(s["q"], s["k"], s["v"], s["g"], s["beta"], s["cu"], w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                   initial_state=w.initial_state, state=w.state, state_indices=w.state_indices,
                   chunk_states=w.return_chunk_states, threads=threads)


def oracle_fraction(oracle, w, budget_s: float, threads: int) -> float:
    """The token fraction whose all-heads sample takes about budget_s on the host cores
    (calibrated on a small probe; the oracle's cost is linear in the tokens)."""
    f = min(1.0, 256.0 / max(max(w.lengths), 1))
    s = oracle_sample(w, f)
    t0 = time.perf_counter()
    _oracle_run(oracle, w, s, threads)
    el = max(time.perf_counter() - t0, 1e-4)
    return min(1.0, f * budget_s / el)


def cpu_oracle_baseline(w, budget_s: float):
    """The oracle as it stands on this host's cores over a bounded sample of the workload."""
    import oracle

    threads = oracle.oracle_threads()
    frac = oracle_fraction(oracle, w, budget_s, threads)
    s = oracle_sample(w, frac)
    t0 = time.perf_counter()
    _oracle_run(oracle, w, s, threads)
    el = time.perf_counter() - t0
    return {"value": s["T"] / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"all {w.H} heads, first {frac:.4f} of each sequence ({s['T']} of {w.T} tokens), "
                      f"one run, {el:.1f} s"}


def run_reference(args, w, rank):
    """Reference arm: the float64 oracle on the host cores, timed on the same kind of sample as
    the CPU baseline (all heads, a prefix of every sequence), one sample per step."""
    import oracle

    if rank != 0:
        return
    threads = oracle.oracle_threads()
    total_steps = args.steps + args.warmup
    per_step_budget = max(0.05, min(5.0, 150.0 / max(total_steps, 1)))
    frac = oracle_fraction(oracle, w, per_step_budget, threads)
    s = oracle_sample(w, frac)
    times = []
    for i in range(total_steps):
        t0 = time.perf_counter()
        _oracle_run(oracle, w, s, threads)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    el = sum(times)
    value = s["T"] * len(times) / el if el > 0 else 0.0
    sample = (f"per step: all {w.H} heads, first {frac:.4f} of each sequence ({s['T']} of {w.T} tokens)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / max(len(times), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**w.describe(), "l2_flush": False}, "impl": "reference",
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------- the GPU legs

def launches_per_call(w) -> int:
    """Kernels one call launches (the library's shape-only plan)."""
    import chunked_gated_deltaproduct_gb300 as pkg
    return pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)["launches"]


def stage_names(w):
    """The three stages the profiled entry point separates by events."""
    import chunked_gated_deltaproduct_gb300 as pkg
    plan = pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)
    if plan["piece_chunks"] > 0:
        scan = "gdp_scan_kernel x2 + gdp_piece_combine_kernel"
    elif plan["segments"] > 1:
        scan = f"gdp_scan_kernel x{plan['segments']} (segmented, WY segments 2.. beside it)"
    else:
        scan = "gdp_scan_kernel"
    wy = "gdp_wy_kernel" if plan["segments"] == 1 else "gdp_wy_kernel (segment 1)"
    return ["gdp_desc_kernel", wy, scan]


class Call:
    """Device tensors and arguments of one workload's call."""

    def __init__(self, pkg, w, dev):
        self.w = w
        self.q, self.k, self.v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
        self.g = None if w.g is None else w.g.to(dev)
        self.beta = None if w.beta is None else w.beta.to(dev)
        self.cu = w.cu_seqlens.to(dev)
        self.init = None if w.initial_state is None else w.initial_state.to(dev)
        self.cache = None if w.state is None else w.state.to(dev)
        self.sidx = None if w.state_indices is None else w.state_indices.to(dev)
        self.out = torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=dev)
        self.fin = torch.empty((w.N, w.H, w.d, w.d), dtype=torch.float32, device=dev) if (
            w.output_final_state and self.cache is None) else None
        self.cs = torch.zeros((pkg.gdp_nt_pad(w.T, w.N), w.H, w.d, w.d), dtype=torch.float32, device=dev) if (
            w.return_chunk_states) else None
        self.ci = self.cid = self.co = None
        if w.prebuilt_descriptors:
            self.ci, self.cid, self.co = pkg.gdp_build_descriptors(self.cu, w.T, w.M)
        self.ws = pkg.alloc_workspace(w.T, w.N, w.H, w.d, w.d, w.M, dev)
        self.args = pkg.make_args(self.q, self.k, self.v, self.g, self.beta, self.cu, w.M, w.scale, self.init,
                                  self.cache, self.sidx, self.out, self.fin, self.cs, self.ci, self.cid, self.co,
                                  None, None, w.use_qk_l2norm, self.ws, None)

    def inputs(self):
        return [t for t in (self.q, self.k, self.v, self.g, self.beta, self.cu, self.init, self.cache, self.sidx)
                if t is not None]

    def outputs(self):
        return [t for t in (self.out, self.fin, self.cs, self.cache) if t is not None]


def time_call(pkg, c, stream, flush, steps, warmup, clk_folder=None, sample_clocks=False):
    """Plain calls (events around each, L2 flushed before each), then the same number of calls
    through the profiled entry point (events between the stages).  Returns step times (ms), the
    mean per-stage times (ms), the profiled step time and the clock summary."""
    sid = stream.cuda_stream

    def new_events():
        # torch creates the CUDA event lazily at its first record(); record once so the raw
        # handle exists and torch accepts elapsed_time(); the library then re-records it.
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in evs:
            e.record(stream)
        return evs

    def step_profiled(evs):
        with torch.cuda.stream(stream):
            flush.zero_()
        pkg.gdp_prefill_varlen_profiled(c.args, evs, sid)

    def step_plain(e0, e1):
        with torch.cuda.stream(stream):
            flush.zero_()
        e0.record(stream)
        pkg.gdp_prefill_varlen(c.args, sid)
        e1.record(stream)

    def pair():
        return [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    for _ in range(warmup):
        step_plain(*pair())
        step_profiled(new_events())
    torch.cuda.synchronize()
    plain = [pair() for _ in range(steps)]
    clk = None
    t_wall = 0.0
    if sample_clocks:
        with ClockSampler(torch.cuda.current_device(), clk_folder) as sampler:
            w0 = time.perf_counter()
            for s in range(steps):
                step_plain(*plain[s])
            torch.cuda.synchronize()
            t_wall = time.perf_counter() - w0
        clk = sampler.summary()
    else:
        for s in range(steps):
            step_plain(*plain[s])
        torch.cuda.synchronize()
    step_ms = [e0.elapsed_time(e1) for e0, e1 in plain]
    events = [new_events() for _ in range(steps)]
    for s in range(steps):
        step_profiled(events[s])
    torch.cuda.synchronize()
    stage = [[ev[i].elapsed_time(ev[i + 1]) for i in range(3)] for ev in events]
    stage_ms = [statistics.fmean(x[i] for x in stage) for i in range(3)]
    prof_ms = statistics.fmean(ev[0].elapsed_time(ev[3]) for ev in events)
    return step_ms, stage_ms, prof_ms, clk, t_wall


def roofline_of(w, step_ms_mean, stage_ms, names, workload_id):
    """Whole-call and dominant-stage fractions of the HBM roofline (algorithmic bytes over the
    measured time; every workload is HBM-bound by its algorithmic count)."""
    peak, src = measured_peaks()
    ab = alg_bytes(w)
    dom = max(range(3), key=lambda i: stage_ms[i])
    stage_gbs = ab / (stage_ms[dom] / 1e3) / 1e9
    step_gbs = ab / (step_ms_mean / 1e3) / 1e9
    tr = NCU_TRAFFIC.get((names[dom], workload_id))
    traffic = tr["bytes_per_call"] if (tr and tr["sha"] == sources_sha(tr["sources"])) else None
    return {"bound": "hbm", "kernel": names[dom], "achieved": stage_gbs, "peak": peak, "peak_source": src,
            "unit": "GB/s", "frac": stage_gbs / peak, "traffic": traffic, "alg_bytes_per_launch": ab,
            "kernel_ms": stage_ms[dom], "step_achieved": step_gbs, "step_frac": step_gbs / peak,
            "roofline_us": ab / (peak * 1e9) * 1e6, "alg_gflop_per_step": alg_flops(w) / 1e9}


def measure_graph(pkg, w, dev, stream, flush, replays=50, warmup=10):
    """A CUDA-graph replay of one call (prebuilt descriptors, the state cache in place): median
    of `replays` replays after `warmup`, the L2 flushed outside the graph before each.  Replays
    keep updating the cache in place (beta in (0, 1) and unit-norm k keep it bounded)."""
    c = Call(pkg, w, dev)
    sid = stream.cuda_stream
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        graph.capture_begin()
        pkg.gdp_prefill_varlen(c.args, sid)
        graph.capture_end()
    torch.cuda.synchronize()
    times = []
    for i in range(warmup + replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
        e1.synchronize()
        if i >= warmup:
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    peak, src = measured_peaks()
    ab = alg_bytes(w)
    live = int((w.state_indices >= 0).sum()) if w.state_indices is not None else w.N
    live_tokens = sum(L for L, s in zip(w.lengths, w.state_indices.tolist()) if s >= 0) if (
        w.state_indices is not None) else w.T
    del graph, c
    return {"workload": w.name, "timing": f"CUDA-graph replay, median of {replays} after {warmup}, L2 flushed",
            "ms_per_call": ms, "tokens_per_s": w.T / (ms / 1e3), "tokens": w.T,
            "live_tokens_per_s": live_tokens / (ms / 1e3), "live_sequences": live,
            "alg_bytes": ab, "achieved_gbs": ab / (ms / 1e3) / 1e9, "frac": ab / (ms / 1e3) / 1e9 / peak,
            "roofline_us": ab / (peak * 1e9) * 1e6, "launches_per_call": launches_per_call(w)}


def measure_decode(pkg, dev, flush, stream, steps=50, warmup=5):
    """The decode step (one token per sequence, state cache in place) on a serving batch shaped
    like the serving workload: 64 sequences, H=16, d=128, M=4, a 128-slot cache with 8 padding
    entries.  Device time per step with the L2 flushed between steps; algorithmic bytes = the
    live cache slots read and written + the token's q, M k/v rows, gate, M betas and o."""
    wd = make_custom([1] * 64, 16, 128, 4, seed=2024, cache_slots=128, cache_sigma=0.1, padding_slots=8)
    q, k, v, g, b = (t.to(dev) for t in (wd.q, wd.k, wd.v, wd.g, wd.beta))
    cache, sidx = wd.state.to(dev), wd.state_indices.to(dev)
    out = torch.empty((wd.N, wd.H, wd.d), dtype=torch.bfloat16, device=dev)
    a = pkg.decode_args(q, k, v, g, b, wd.M, wd.scale, None, cache, sidx, out, None, False, None)
    sid = stream.cuda_stream
    times = []
    for s in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            pkg.gdp_decode_step(a, sid)
            e1.record(stream)
        e1.synchronize()
        if s >= warmup:
            times.append(e0.elapsed_time(e1))
    live = int((wd.state_indices >= 0).sum())
    d, M, H, N = wd.d, wd.M, wd.H, wd.N
    ab = live * H * d * d * 4 * 2 + N * H * (2 * d + M * 4 * d + 4 + 4 * M + 2 * d)
    ms = statistics.median(times)
    peak, src = measured_peaks()
    gbs = ab / (ms / 1e3) / 1e9
    return {"workload": "decode: 64 seqs x 1 token, H16 d128 M4, cache 128 slots (8 padding)",
            "us_per_step": 1e3 * ms, "tokens_per_s": N / (ms / 1e3), "alg_bytes": ab, "achieved_gbs": gbs,
            "peak_gbs": peak, "frac": gbs / peak, "peak_source": src, "steps": steps, "l2_flush": True}


def rank_seed(workload: int, rank: int):
    """Input seed of a rank: rank 0 draws the workload's own inputs, every other rank an
    independent batch of the same shape (replicas, weak scaling)."""
    return 1000 + workload + 7919 * rank if rank else None


def max_over_ranks(x: float, dist, device) -> float:
    """The largest value of x over the ranks of the process group (x itself without one)."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def backward_alg_bytes(w, with_dfin: bool) -> int:
    """Algorithmic bytes of one backward call: q, k, v, d_output (bf16), g, beta (fp32) and the
    initial state / final-state gradient (fp32) read once; dq, dk, dv, dg, dbeta and the
    initial-state gradient (fp32) written once."""
    d, M, H, T, N = w.d, w.M, w.H, w.T, w.N
    rd = T * H * (2 * d * (2 + 2 * M) + 4 + 4 * M)
    wr = T * H * (4 * d * (1 + 2 * M) + 4 + 4 * M)
    st = N * H * d * d * 4
    return int(rd + wr + (st if w.initial_state is not None else 0) * 2 + (st if with_dfin else 0))


def backward_launches(w) -> int:
    """Kernels one backward call launches: the forward recompute, two memsets (the sums and
    dbeta), the reverse scan, the per-chunk gradients, the row pass and the decay pass."""
    return launches_per_call(w) + 2 + 4


def measure_backward(pkg, dev, flush, stream, w, steps=5, warmup=3):
    """The backward pass of the same workload: upstream gradients d_output (bf16) and
    d_final_state (fp32) drawn by gdp_workloads.make_cotangents; device time per call with the
    L2 flushed between calls."""
    from gdp_workloads import make_cotangents

    d_out, d_fin = make_cotangents(w, seed=1, dfin_sigma=0.5)
    dd = lambda x: None if x is None else x.to(dev)
    q, k, v, g, beta, init = (dd(t) for t in (w.q, w.k, w.v, w.g, w.beta, w.initial_state))
    cu, dout, dfin = w.cu_seqlens.to(dev), d_out.to(dev), d_fin.to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    T, H, d, M, N = w.T, w.H, w.d, w.M, w.N
    dq, dk, dv = torch.empty((T, H, d), **f32), torch.empty((T * M, H, d), **f32), torch.empty((T * M, H, d), **f32)
    dg, db = torch.empty((T, H), **f32), torch.empty((T * M, H), **f32)
    dinit = torch.empty((N, H, d, d), **f32) if init is not None else None
    ws = torch.empty(pkg.gdp_backward_workspace_bytes(T, N, H, d, d, M), dtype=torch.uint8, device=dev)
    fa = pkg.make_args(q, k, v, g, beta, cu, M, w.scale, init, None, None, None, None, None, None, None, None, None,
                       None, w.use_qk_l2norm, None, None)
    b = pkg.backward_args(fa, dout, dfin, dq, dk, dv, dg, db, dinit, ws)
    sid = stream.cuda_stream
    times = []
    for s in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            pkg.gdp_prefill_varlen_backward(b, sid)
            e1.record(stream)
        e1.synchronize()
        if s >= warmup:
            times.append(e0.elapsed_time(e1))
    ms = statistics.fmean(times)
    ab = backward_alg_bytes(w, True)
    peak, src = measured_peaks()
    gbs = ab / (ms / 1e3) / 1e9
    del ws, b, fa
    return {"workload": w.name, "ms_per_call": ms, "tokens_per_s": T / (ms / 1e3), "alg_bytes": ab,
            "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak, "peak_source": src, "steps": steps,
            "l2_flush": True, "launches_per_call": backward_launches(w),
            "note": "includes the forward recompute (the backward keeps nothing from a forward call)"}


def time_fused(pkg, c, stream, flush, steps=10, warmup=3):
    """Mean ms per call of the same arguments through gdp_prefill_varlen_fused (L2 flushed), or
    None when the fused kernel does not serve the workload."""
    w = c.w
    if pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M) is None:
        return None
    sid = stream.cuda_stream
    times = []
    for s in range(warmup + steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            pkg.gdp_prefill_varlen_fused(c.args, sid)
            e1.record(stream)
        e1.synchronize()
        if s >= warmup:
            times.append(e0.elapsed_time(e1))
    ms = statistics.fmean(times)
    peak, _ = measured_peaks()
    return {"ms_per_call": ms, "tokens_per_s": w.T / (ms / 1e3),
            "step_frac": alg_bytes(w) / (ms / 1e3) / 1e9 / peak, "steps": steps}


def measure_other(pkg, wid, dev, stream, flush, steps=20, warmup=5):
    """One of the other benchmark configurations: plain calls (or a graph replay for the
    serving step), with the same roofline arithmetic as the headline."""
    w = make_workload(wid)
    if w.graph:
        return measure_graph(pkg, w, dev, stream, flush)
    c = Call(pkg, w, dev)
    step_ms, stage_ms, prof_ms, _, _ = time_call(pkg, c, stream, flush, steps, warmup)
    names = stage_names(w)
    rf = roofline_of(w, statistics.fmean(step_ms), stage_ms, names, wid)
    fused = time_fused(pkg, c, stream, flush)
    del c
    return {"workload": w.name, "timing": f"plain calls, mean of {steps} after {warmup}, L2 flushed",
            "ms_per_call": statistics.fmean(step_ms), "tokens_per_s": w.T / (statistics.fmean(step_ms) / 1e3),
            "step_frac": rf["step_frac"], "stage_frac": rf["frac"], "dominant_stage": rf["kernel"],
            "stages_ms": dict(zip(names, stage_ms)), "profiled_ms_per_call": prof_ms,
            "alg_bytes": rf["alg_bytes_per_launch"], "roofline_us": rf["roofline_us"],
            "launches_per_call": launches_per_call(w), "fused_entry_point": fused}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=HEADLINE_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="gdp", choices=["gdp", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the per_workload legs")
    ap.add_argument("--no-fused", action="store_true", help="skip the fused entry point's timing")
    ap.add_argument("--no-decode", action="store_true", help="skip the decode step's timing")
    ap.add_argument("--clocks-dir", default=None, help="folder for the raw clock samples (default: a temp folder)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        dist = dist_mod
        dist.init_process_group("nccl" if args.impl == "gdp" else "gloo")

    w = make_workload(args.workload, seed=rank_seed(args.workload, rank))

    if args.impl == "reference":
        run_reference(args, w, rank)
        if dist:
            dist.destroy_process_group()
        return

    import chunked_gated_deltaproduct_gb300 as pkg

    pkg.load_library()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    c = Call(pkg, w, dev)
    torch.cuda.synchronize()

    if dist:
        dist.barrier()
    step_ms, stage_ms, prof_ms, clk, wall = time_call(pkg, c, stream, flush, args.steps, args.warmup,
                                                       args.clocks_dir, sample_clocks=True)
    if dist:
        dist.barrier()
    total_s = max_over_ranks(sum(step_ms) / 1e3, dist, dev)
    value = world * w.T * args.steps / total_s
    names = stage_names(w)
    rf = roofline_of(w, statistics.fmean(step_ms), stage_ms, names, args.workload)

    fused_head = time_fused(pkg, c, stream, flush) if (rank == 0 and not args.no_fused) else None

    # ---- end to end: pinned host inputs -> device -> call -> host outputs, same stream
    host_in = [t.pin_memory() for t in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.initial_state, w.state,
                                        w.state_indices) if t is not None]
    dev_in = c.inputs()
    dev_out = c.outputs()
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in dev_out]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    sid = stream.cuda_stream
    e2e_ms = []
    for s in range(args.e2e_steps + 2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            flush.zero_()
            e0.record(stream)
            for hsrc, ddst in zip(host_in, dev_in):
                ddst.copy_(hsrc, non_blocking=True)
            pkg.gdp_prefill_varlen(c.args, sid)
            for dsrc, hdst in zip(dev_out, host_out):
                hdst.copy_(dsrc, non_blocking=True)
            e1.record(stream)
        e1.synchronize()
        if s >= 2:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e_value = world * w.T / (statistics.fmean(e2e_ms) / 1e3)
    del host_in, host_out, c
    torch.cuda.empty_cache()

    others = {}
    if rank == 0 and not args.no_others:
        for wid in PER_WORKLOAD:
            if wid != args.workload:
                others[str(wid)] = measure_other(pkg, wid, dev, stream, flush)
                torch.cuda.empty_cache()
    decode = measure_decode(pkg, dev, flush, stream) if (rank == 0 and not args.no_decode) else None
    bwd = measure_backward(pkg, dev, flush, stream, w) if (rank == 0 and not args.no_backward) else None

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline and world == 1:
            cpu = cpu_oracle_baseline(w, args.cpu_budget_s)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16/tf32 MMA, f32 state", "data": "synthetic",
            "config": {**w.describe(), "l2_flush": True, "flush_bytes": flush.numel()},
            "roofline": rf,
            "step_roofline": {"achieved": rf["step_achieved"], "frac": rf["step_frac"], "unit": "GB/s",
                              "scope": "whole call (all kernels), algorithmic bytes / mean step time"},
            "stages_ms": dict(zip(names, stage_ms)),
            "profiled_ms_per_step": prof_ms,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": statistics.fmean(e2e_ms)},
            "gpu_launches": launches_per_call(w) * args.steps,
            "clocks": clk,
            "per_workload": others,
            "fused_entry_point": fused_head,
            "decode_step": decode,
            "backward": bwd,
            "wall_s_timed": wall,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
