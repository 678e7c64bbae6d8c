"""Seeded synthetic inputs for the chunked Gated DeltaProduct prefill.

Serves the tests, the smoke check and the bench, for both the CUDA path and
the oracle.  It holds none of the method's arithmetic: it only draws random
tensors with the shapes, dtypes and value distributions of the five workloads
below and packs them into the THD / expanded-stream layout of the tensor
contract (FlashInfer page "flashinfer.gdp_prefill.chunk_gated_delta_product",
parameters q, k, v, g, beta, initial_state, cu_seqlens; Megatron page
"core.ssm.ops.gdp.chunk", parameters state, state_indices).

Recipe (every tensor drawn on the CPU from one torch.Generator seeded with
1000 + workload id, in the order lengths, q, k, v, g, beta, state,
state_indices):
  * q, k, v ~ N(0, 1) in fp32; rows are L2-normalised per (row, head) in fp32
    when the workload says "normalised", then cast to bf16;
  * g = -U(0, a) fp32, the natural log of alpha = exp(-U(0, a));
  * beta = sigmoid(N(0, 1)) fp32 on the expanded stream;
  * states sigma * N(0, 1) fp32, V-major [., H, V, K].

Input variants of the same contract (FlashInfer page, parameters q, k, v, g,
beta, initial_state), all off by default so that the draws above are
unchanged: q / k / v (and so the output) in float16; the gate drawn as alpha =
exp(-U(0, a)) itself (linear space) instead of its log; g and beta rounded to
bfloat16 or float16; the initial state rounded to bfloat16; q, k and v with
fewer heads than the H state heads (each count divides H; the per-head draws
simply have that many heads).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

CHUNK = 64


@dataclass
class Workload:
    name: str
    lengths: list
    H: int
    d: int
    M: int
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    g: torch.Tensor | None
    beta: torch.Tensor | None
    cu_seqlens: torch.Tensor
    scale: float
    use_qk_l2norm: bool = False
    initial_state: torch.Tensor | None = None
    state: torch.Tensor | None = None
    state_indices: torch.Tensor | None = None
    output_final_state: bool = True
    return_chunk_states: bool = False
    prebuilt_descriptors: bool = False
    graph: bool = False
    g_is_alpha: bool = False
    meta: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(sum(self.lengths))

    @property
    def N(self) -> int:
        return len(self.lengths)

    @property
    def NT(self) -> int:
        return sum((L + CHUNK - 1) // CHUNK for L in self.lengths)

    @property
    def NTdp(self) -> int:
        return sum((L * self.M + CHUNK - 1) // CHUNK for L in self.lengths)

    def describe(self) -> dict:
        return {"workload": self.name, "N": self.N, "T": self.T, "H": self.H, "head_size": self.d,
                "num_householder": self.M, "lengths": (self.lengths if self.N <= 8 else
                                                       f"{self.N} seqs, min {min(self.lengths)}, max {max(self.lengths)}")}


def _normal(gen, shape):
    return torch.randn(*shape, generator=gen, dtype=torch.float32)


def _rows(gen, rows, H, d, normalise, dtype=torch.bfloat16):
    x = _normal(gen, (rows, H, d))
    if normalise:
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    return x.to(dtype)


def make_custom(lengths, H, d, M, *, seed=0, normalised=True, use_qk_l2norm=False,
                decay=0.1, init_sigma=0.0, cache_slots=0, cache_sigma=0.1, padding_slots=0,
                chunk_states=False, with_g=True, with_beta=True, name="custom",
                prebuilt_descriptors=False, graph=False, scale=None,
                qkv_dtype=torch.bfloat16, hq=None, hk=None, hv=None, g_is_alpha=False,
                g_dtype=torch.float32, beta_dtype=torch.float32, state_dtype=torch.float32) -> Workload:
    """A workload of the given shape drawn with the recipe of this module (H state heads;
    hq / hk / hv: head counts of q / k / v, default H)."""
    gen = torch.Generator().manual_seed(int(seed))
    lengths = [int(x) for x in lengths]
    T, N = sum(lengths), len(lengths)
    q = _rows(gen, T, hq or H, d, normalised, qkv_dtype)
    k = _rows(gen, T * M, hk or H, d, normalised, qkv_dtype)
    v = _rows(gen, T * M, hv or H, d, False, qkv_dtype)
    g = -torch.rand(T, H, generator=gen, dtype=torch.float32) * decay if with_g else None
    if g is not None:
        g = (torch.exp(g) if g_is_alpha else g).to(g_dtype)
    beta = torch.sigmoid(_normal(gen, (T * M, H))) if with_beta else None
    if beta is not None:
        beta = beta.to(beta_dtype)
    init = state = sidx = None
    if cache_slots:
        state = _normal(gen, (cache_slots, H, d, d)) * cache_sigma
        perm = torch.randperm(cache_slots, generator=gen)[:N].to(torch.int32)
        if padding_slots:
            pos = torch.randperm(N, generator=gen)[:padding_slots]
            perm[pos] = -1
        sidx = perm
    elif init_sigma > 0:
        init = (_normal(gen, (N, H, d, d)) * init_sigma).to(state_dtype)
    cu = torch.zeros(N + 1, dtype=torch.int32)
    if N:
        cu[1:] = torch.cumsum(torch.tensor(lengths, dtype=torch.int64), 0).to(torch.int32)
    return Workload(name=name, lengths=lengths, H=H, d=d, M=M, q=q, k=k, v=v, g=g, beta=beta,
                    cu_seqlens=cu, scale=(1.0 / math.sqrt(d)) if scale is None else scale,
                    use_qk_l2norm=use_qk_l2norm, initial_state=init, state=state,
                    state_indices=sidx, output_final_state=(state is None),
                    return_chunk_states=chunk_states, prebuilt_descriptors=prebuilt_descriptors,
                    graph=graph, g_is_alpha=g_is_alpha)


def _loguniform_lengths(gen, n, lo, hi):
    u = torch.rand(n, generator=gen, dtype=torch.float64)
    x = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
    return [int(min(max(math.floor(float(t)), lo), hi)) for t in x]


WORKLOADS = {
    1: "gdn-n1-L256-H2-d64",
    2: "gdp-n2-varlen4-H8-d128-chunkstates",
    3: "gdp-n3-8x4096-H16-d128-l2norm",
    4: "gdp-n2-L65536-H32-d128-chunkstates",
    5: "gdp-n4-64seq-loguniform-H16-d128-statecache-graph",
}


def make_workload(wid: int, seed: int | None = None) -> Workload:
    """The five synthetic workloads (sizes of the benchmark configurations)."""
    s = 1000 + wid if seed is None else seed
    name = WORKLOADS[wid]
    if wid == 1:
        return make_custom([256], 2, 64, 1, seed=s, decay=0.1, name=name)
    if wid == 2:
        return make_custom([100, 257, 64, 1000], 8, 128, 2, seed=s, decay=0.05, init_sigma=0.1,
                           chunk_states=True, name=name)
    if wid == 3:
        return make_custom([4096] * 8, 16, 128, 3, seed=s, normalised=False, use_qk_l2norm=True,
                           decay=0.1, name=name)
    if wid == 4:
        return make_custom([65536], 32, 128, 2, seed=s, decay=0.02, init_sigma=0.05,
                           chunk_states=True, name=name)
    if wid == 5:
        gen = torch.Generator().manual_seed(s)
        lengths = _loguniform_lengths(gen, 64, 16, 8192)
        # the remaining tensors come from a second stream so that the lengths
        # stay the same whatever the other shapes are
        w = make_custom(lengths, 16, 128, 4, seed=s + 7919, decay=0.1, cache_slots=128,
                        cache_sigma=0.1, padding_slots=8, name=name, prebuilt_descriptors=True,
                        graph=True)
        return w
    raise KeyError(wid)


def make_cotangents(w: Workload, *, seed=0, dfin_sigma=1.0, d_final_state=True, quantum=None):
    """Seeded upstream gradients for the backward pass of workload ``w``: d_output [T, H, V]
    bf16 ~ N(0, 1) (the type of the output) and d_final_state [N, H, V, K] fp32 ~ dfin_sigma N(0, 1)
    (None when ``d_final_state`` is False).  ``quantum``: when given, g, beta and the initial
    state of ``w`` are replaced by their values rounded to multiples of it (a grid on which
    finite-difference steps that are multiples of ``quantum`` stay exact in fp32)."""
    gen = torch.Generator().manual_seed(int(seed) + 77)
    d_out = _normal(gen, (w.T, w.H, w.d)).to(torch.bfloat16)
    d_fin = _normal(gen, (w.N, w.H, w.d, w.d)) * dfin_sigma if d_final_state else None
    if quantum is not None:
        def snap(x):
            return None if x is None else (torch.round(x.double() / quantum) * quantum).to(x.dtype)
        w.g, w.beta, w.initial_state = snap(w.g), snap(w.beta), snap(w.initial_state)
    return d_out, d_fin
