"""Runs a few prefill calls of a reduced, benchmark-shaped case: the command the committed ncu
summaries under profiles/ were captured on (the full-size workloads are too large for a
multi-pass capture).

    python -m chunked_gated_deltaproduct_gb300.profile_case {w3|w4|w2|decode|desc|bwd} [--calls N] [--fused]

w3: 8 sequences x 1024 tokens, H=16, d=128, M=3, unnormalised q/k with in-kernel L2 norm (the
    8 x 4096 batch cut to a quarter of its length); w4: one sequence of 12288 tokens, H=32, d=128,
    M=2, initial state and chunk states (the 65536-token sequence cut to its first six segments,
    the segmented plan); w2: the four-sequence varlen batch at full size; decode: the decode step
    of the serving batch; desc: the descriptor kernel alone over 3000 sequences; bwd: the backward
    pass of the 65536-token shape cut to 4096 tokens (H=32, d=128, M=2, initial state).
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    import chunked_gated_deltaproduct_gb300 as pkg
    from gdp_workloads import make_custom, make_workload

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["w2", "w3", "w4", "decode", "desc", "bwd"])
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--fused", action="store_true")
    a = ap.parse_args()
    pkg.load_library()
    dev = torch.device("cuda:0")
    if a.case == "desc":
        import numpy as np
        lengths = [(7 * i) % 500 + 1 for i in range(3000)]
        cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32, device=dev)
        for _ in range(a.calls):
            pkg.gdp_build_descriptors(cu, int(sum(lengths)), 2)
        torch.cuda.synchronize()
        return
    if a.case == "decode":
        w = make_custom([1] * 64, 16, 128, 4, seed=2024, cache_slots=128, cache_sigma=0.1, padding_slots=8)
        q, k, v, g, b = (t.to(dev) for t in (w.q, w.k, w.v, w.g, w.beta))
        cache, sidx = w.state.to(dev), w.state_indices.to(dev)
        out = torch.empty((w.N, w.H, w.d), dtype=torch.bfloat16, device=dev)
        args = pkg.decode_args(q, k, v, g, b, w.M, w.scale, None, cache, sidx, out, None, False, None)
        for _ in range(a.calls):
            pkg.gdp_decode_step(args)
        torch.cuda.synchronize()
        return
    if a.case == "bwd":
        from gdp_workloads import make_cotangents

        w = make_custom([4096], 32, 128, 2, seed=1004, decay=0.02, init_sigma=0.05)
        d_out, d_fin = make_cotangents(w, seed=1, dfin_sigma=0.5)
        dd = lambda x: None if x is None else x.to(dev)
        for _ in range(a.calls):
            pkg.chunk_gated_delta_product_backward(dd(w.q), dd(w.k), dd(w.v), dd(w.g), dd(w.beta), w.cu_seqlens.to(dev),
                                                   w.M, dd(d_out), scale=w.scale, initial_state=dd(w.initial_state),
                                                   d_final_state=dd(d_fin))
        torch.cuda.synchronize()
        return
    if a.case == "w2":
        w = make_workload(2)
    elif a.case == "w3":
        w = make_custom([1024] * 8, 16, 128, 3, seed=1003, normalised=False, use_qk_l2norm=True, decay=0.1)
    else:
        w = make_custom([12288], 32, 128, 2, seed=1004, decay=0.02, init_sigma=0.05, chunk_states=True)
    d = {n: (None if t is None else t.to(dev)) for n, t in
         (("q", w.q), ("k", w.k), ("v", w.v), ("g", w.g), ("beta", w.beta), ("init", w.initial_state))}
    cu = w.cu_seqlens.to(dev)
    for _ in range(a.calls):
        pkg.chunk_gated_delta_product(d["q"], d["k"], d["v"], d["g"], d["beta"], cu, w.M, w.scale,
                                      initial_state=d["init"], output_final_state=True,
                                      use_qk_l2norm_in_kernel=w.use_qk_l2norm,
                                      return_chunk_states=w.return_chunk_states, fused=a.fused)
    torch.cuda.synchronize()


if __name__ == "__main__":
    main()
