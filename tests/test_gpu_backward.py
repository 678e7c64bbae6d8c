"""GPU parity of the backward pass (gdp_prefill_varlen_backward) against the float64
oracle's reverse mode of the recurrence.

Every gradient of q, k, v, beta and the initial state is compared per head with a
relative L2 error bound of 5e-3 -- the bound of the forward output; the decay gradient,
a sum whose terms can be far larger than the result, with the same factor against the
magnitude of those terms (_dg_scale).  The GPU path uses tf32
tensor-core products with fp32 accumulation (relative rounding of 2^-11 per operand),
and its dq, dk, dbeta and dg are sums of per-slice shares; 5e-3 leaves room for the
~1e-3 these accumulate to.  Cases cover ragged chunk tails, token rows that straddle
chunks (M = 3), the gated delta rule (M = 1, d = 64), the in-kernel L2 norm, no decay
and no beta, chunks whose decay takes the unscaled ("slow") image path, empty
sequences, a long single sequence, and the segmented forward recompute.
"""
import numpy as np
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_cotangents, make_custom
from tests._parity import per_head_rel

pytestmark = pytest.mark.gpu

TOL_GRAD_REL = 5e-3


def _check(name, gpu, ref, head_axis):
    g = gpu.detach().double().cpu().numpy()
    rel, den = per_head_rel(g, ref, head_axis)
    ok = np.where(den == 0, rel <= 1e-6, rel <= TOL_GRAD_REL)
    assert ok.all(), f"{name}: worst head rel L2 {rel.max():.3e} (head {int(np.argmax(rel))})"
    return float(rel.max())


def _dg_scale(w, d_out, d_fin, ref):
    """Per (token, head) magnitude of the terms summed into dg_t (the decay gradient needs no
    state: dg_t = <dS_T, S_T> + sum_{t' >= t} (do_t' . o_t' - sum_j dv_j . v_j) over the rest
    of the sequence): c_t = |dS_T| |S_T| + sum_{t' >= t} (|do_t'| |o_t'| + sum_j |dv_j| |v_j|).
    Each term reaches the GPU with the relative error of the state and output it is built from
    (the forward's own bound is 2e-3 on states), so the error of dg is bounded relative to c,
    not to dg itself: |dg| can be far smaller than its terms (here the constant <dS_T, S_T> of
    a random final-state gradient dominates)."""
    M = w.M
    do = d_out.double().numpy()
    a = np.linalg.norm(do, axis=-1) * np.linalg.norm(ref["o"], axis=-1)  # [T, H]
    v = w.v.double().numpy()
    b = (np.linalg.norm(ref["dv"], axis=-1) * np.linalg.norm(v, axis=-1)).reshape(w.T, M, -1).sum(1)
    x = a + b
    c = np.zeros_like(x)
    cu = w.cu_seqlens.tolist()
    for i in range(w.N):
        s0, s1 = cu[i], cu[i + 1]
        base = 0.0
        if d_fin is not None:
            base = np.linalg.norm(d_fin.double().numpy()[i], axis=(-1, -2)) * np.linalg.norm(
                ref["final_state"][i], axis=(-1, -2))
        c[s0:s1] = base + np.cumsum(x[s0:s1][::-1], 0)[::-1]
    return c


def _check_dg(gpu, ref, scale):
    g = gpu.detach().double().cpu().numpy()
    err = np.linalg.norm(g - ref, axis=0)
    bound = TOL_GRAD_REL * np.linalg.norm(scale, axis=0)
    assert (err <= bound).all(), f"dg: error {err} above {bound}"
    return float((err / np.maximum(np.linalg.norm(ref, axis=0), 1e-300)).max())


def _run(w, dev, d_out, d_fin):
    dd = lambda x: None if x is None else x.to(dev)
    res = pkg.chunk_gated_delta_product_backward(
        dd(w.q), dd(w.k), dd(w.v), dd(w.g), dd(w.beta), w.cu_seqlens.to(dev), w.M, dd(d_out), scale=w.scale,
        initial_state=dd(w.initial_state), d_final_state=dd(d_fin), use_qk_l2norm_in_kernel=w.use_qk_l2norm)
    torch.cuda.synchronize()
    return res


def _compare(w, dev, d_out, d_fin):
    res = _run(w, dev, d_out, d_fin)
    ref = oracle.backward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, d_out,
                          use_qk_l2norm=w.use_qk_l2norm, initial_state=w.initial_state, d_final_state=d_fin)
    errs = {}
    errs["dq"] = _check("dq", res["dq"], ref["dq"], 1)
    errs["dk"] = _check("dk", res["dk"], ref["dk"], 1)
    errs["dv"] = _check("dv", res["dv"], ref["dv"], 1)
    errs["dbeta"] = _check("dbeta", res["dbeta"], ref["dbeta"], 1)
    if w.g is not None:
        errs["dg"] = _check_dg(res["dg"], ref["dg"], _dg_scale(w, d_out, d_fin, ref))
    if w.initial_state is not None:
        errs["d_initial_state"] = _check("d_initial_state", res["d_initial_state"], ref["d_initial_state"], 1)
    return errs


CASES = {
    "varlen_m2_tails": dict(lengths=[100, 257, 64, 300], H=4, d=128, M=2, init_sigma=0.1),
    "straddle_m3_l2norm": dict(lengths=[37, 64, 130], H=2, d=128, M=3, normalised=False, use_qk_l2norm=True,
                               init_sigma=0.1),
    "gdn_m1_d64": dict(lengths=[256], H=2, d=64, M=1),
    "m4_no_decay_no_beta": dict(lengths=[50, 200], H=2, d=128, M=4, with_g=False, with_beta=False,
                                init_sigma=0.05),
    "slow_decay": dict(lengths=[300, 90], H=2, d=128, M=2, decay=3.0, init_sigma=0.1),
    "empty_sequences": dict(lengths=[0, 70, 0, 5], H=2, d=64, M=2, init_sigma=0.1),
    "long_chain": dict(lengths=[2000], H=2, d=128, M=2, decay=0.05, init_sigma=0.1),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_parity(cuda_device, case):
    kw = dict(CASES[case])
    lengths = kw.pop("lengths")
    w = make_custom(lengths, kw.pop("H"), kw.pop("d"), kw.pop("M"), seed=100 + sorted(CASES).index(case), **kw)
    d_out, d_fin = make_cotangents(w, seed=7, dfin_sigma=0.5)
    _compare(w, cuda_device, d_out, d_fin)


# The per-chunk gradients run on the tensor cores for head size 128 with at most 32 readout rows per
# expanded chunk (two or more updates per token) and on warp-level MMAs otherwise; both kernels
# against the oracle at the shapes that pick them.
PATH_CASES = {
    "warp_mma_d128_m1": (dict(lengths=[130, 64, 7], H=2, d=128, M=1, init_sigma=0.1), 201),
    "tensor_core_qpad16_m5_l2norm": (dict(lengths=[77, 30, 150], H=2, d=128, M=5, normalised=False,
                                          use_qk_l2norm=True, init_sigma=0.1), 202),
    "tensor_core_single_chunks": (dict(lengths=[1, 31, 32, 33], H=3, d=128, M=2, init_sigma=0.1), 203),
}


@pytest.mark.parametrize("case", sorted(PATH_CASES))
def test_backward_kernel_paths(cuda_device, case):
    kw, seed = PATH_CASES[case]
    kw = dict(kw)
    lengths = kw.pop("lengths")
    w = make_custom(lengths, kw.pop("H"), kw.pop("d"), kw.pop("M"), seed=seed, **kw)
    d_out, d_fin = make_cotangents(w, seed=seed + 1, dfin_sigma=0.5)
    _compare(w, cuda_device, d_out, d_fin)


def test_backward_without_final_state_gradient(cuda_device):
    w = make_custom([120, 33], 2, 128, 2, seed=5, init_sigma=0.1)
    d_out, _ = make_cotangents(w, seed=8, d_final_state=False)
    _compare(w, cuda_device, d_out, None)


def test_backward_segmented_recompute(cuda_device):
    """One long sequence over few heads: the forward recompute runs in chunk segments."""
    w = make_custom([12800], 1, 64, 2, seed=9, decay=0.05, init_sigma=0.1)
    d_out, d_fin = make_cotangents(w, seed=10, dfin_sigma=0.5)
    _compare(w, cuda_device, d_out, d_fin)


def test_backward_repeatable_and_graph_capturable(cuda_device):
    """Two calls give identical bits (the kernels use no atomics: every gradient element is
    written once by one thread, in a fixed order), and the call captures into a CUDA graph whose
    replay gives those same bits."""
    w = make_custom([100, 180], 2, 128, 2, seed=11, init_sigma=0.1)
    d_out, d_fin = make_cotangents(w, seed=12)
    a = _run(w, cuda_device, d_out, d_fin)
    b = _run(w, cuda_device, d_out, d_fin)
    for n in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"):
        assert torch.equal(a[n], b[n]), n
    dev = cuda_device
    dd = lambda x: None if x is None else x.to(dev)
    args = [dd(w.q), dd(w.k), dd(w.v), dd(w.g), dd(w.beta), w.cu_seqlens.to(dev), w.M, dd(d_out)]
    kw = dict(scale=w.scale, initial_state=dd(w.initial_state), d_final_state=dd(d_fin))
    ws = torch.empty(pkg.gdp_backward_workspace_bytes(w.T, w.N, w.H, w.d, w.d, w.M), dtype=torch.uint8, device=dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pkg.chunk_gated_delta_product_backward(*args, workspace=ws, **kw)  # warm-up (attributes, lookups)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        out = pkg.chunk_gated_delta_product_backward(*args, workspace=ws, **kw)
    graph.replay()
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"):
        assert torch.equal(out[n], a[n]), n


def test_backward_workload2_full_size(cuda_device):
    """The bench's backward workload at full size (workload 2: N=4, L={100,257,64,1000}, H=8,
    d=128, M=2, initial state), every head, with the bench's upstream gradients."""
    from gdp_workloads import make_workload

    w = make_workload(2)
    d_out, d_fin = make_cotangents(w, seed=1, dfin_sigma=0.5)
    _compare(w, cuda_device, d_out, d_fin)


def test_backward_empty_batch(cuda_device):
    """No tokens at all: the initial-state gradient is the final-state gradient passed through."""
    w = make_custom([0, 0], 2, 64, 2, seed=13, init_sigma=0.1)
    d_out, d_fin = make_cotangents(w, seed=14)
    res = _run(w, cuda_device, d_out, d_fin)
    assert res["dq"].numel() == 0 and res["dv"].numel() == 0
    assert torch.equal(res["d_initial_state"].cpu(), d_fin)
