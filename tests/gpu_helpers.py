"""Shared helpers of the GPU tests: move a workload to the device and run it
through the C ABI (via the thin binding)."""
from __future__ import annotations

import torch

import chunked_gated_deltaproduct_gb300 as pkg


def to_dev(w, dev, cu_dtype=torch.int32):
    return {
        "q": w.q.to(dev), "k": w.k.to(dev), "v": w.v.to(dev),
        "g": None if w.g is None else w.g.to(dev),
        "beta": None if w.beta is None else w.beta.to(dev),
        "cu": w.cu_seqlens.to(cu_dtype).to(dev),
        "init": None if w.initial_state is None else w.initial_state.to(dev),
        "state": None if w.state is None else w.state.to(dev).clone(),
        "sidx": None if w.state_indices is None else w.state_indices.to(dev),
    }


def run(w, dev, d=None, prebuilt=False, status=None, scale=None, **kw):
    """One call through the library (``fused=True``: the fused entry point); returns
    (o, final_state, chunk_states, device tensors)."""
    d = d or to_dev(w, dev)
    ci = cid = co = None
    if prebuilt:
        ci, cid, co = pkg.gdp_build_descriptors(d["cu"], w.T, w.M, device_status=status)
    res = pkg.chunk_gated_delta_product(
        d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale if scale is None else scale,
        initial_state=d["init"], output_final_state=w.output_final_state,
        use_qk_l2norm_in_kernel=w.use_qk_l2norm, chunk_indices=ci, chunk_indices_dp=cid, chunk_offsets=co,
        state=d["state"], state_indices=d["sidx"], return_chunk_states=w.return_chunk_states,
        device_status=status, g_is_alpha=w.g_is_alpha, **kw)
    torch.cuda.synchronize()
    if isinstance(res, tuple):
        o = res[0]
        fin = res[1] if len(res) > 1 else None
        cs = res[2] if len(res) > 2 else None
    else:
        o, fin, cs = res, None, None
    return o, fin, cs, d
