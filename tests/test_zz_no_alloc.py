"""gdp_prefill_varlen_static_scratch: the prefill for callers that cannot
allocate device memory (a plugin inside a runtime that owns all device memory,
or a host program that may not call cudaMalloc in its serving loop).

The entry point is called through the C ABI twice in a row on the same inputs,
once for each of the three ways a call runs (plain, split chains, segmented;
gdp_prefill_plan names which), and each result must equal, bit for bit, the
main entry point's result with a caller-owned workspace: the two run the same
kernels in the same order, only the scratch memory differs.  One call of each
shape is also checked against the float64 oracle with the parity tolerances.
A shape whose scratch need exceeds the static array is rejected before any
launch.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state

pytestmark = pytest.mark.gpu

# (lengths, H, head size, M, the plan the shape takes)
SHAPES = [
    ([5 * i + 3 for i in range(40)], 2, 128, 3, "plain"),
    ([100, 257, 64, 300], 4, 128, 2, "split"),
    ([12288], 1, 128, 2, "segmented"),
    ([100, 257, 64, 300], 4, 64, 1, "split"),
]


def _plan_kind(w):
    plan = pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)
    return "segmented" if plan["segments"] > 1 else ("split" if plan["piece_chunks"] > 0 else "plain")


def _args(w, d, out, fin, cs, workspace):
    return pkg.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale, d["init"], None, None,
                         out, fin, cs, None, None, None, None, None, w.use_qk_l2norm, workspace, None)


@pytest.mark.parametrize("lengths,H,d,M,kind", SHAPES)
def test_static_scratch_matches_caller_workspace(cuda_device, lengths, H, d, M, kind):
    w = make_custom(lengths, H, d, M, seed=77, init_sigma=0.1, chunk_states=True)
    assert pkg.gdp_prefill_workspace_bytes(w.T, w.N, w.H, w.d, w.d, w.M) <= pkg.gdp_static_scratch_bytes()
    assert _plan_kind(w) == kind
    dev = cuda_device
    d = {"q": w.q.to(dev), "k": w.k.to(dev), "v": w.v.to(dev), "g": w.g.to(dev), "beta": w.beta.to(dev),
         "cu": w.cu_seqlens.to(dev), "init": w.initial_state.to(dev)}
    nt = pkg.gdp_nt_pad(w.T, w.N)

    def outputs():
        return (torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=dev),
                torch.empty((w.N, w.H, w.d, w.d), dtype=torch.float32, device=dev),
                torch.zeros((nt, w.H, w.d, w.d), dtype=torch.float32, device=dev))

    # reference: the main entry point with a caller-owned workspace
    ro, rf, rc = outputs()
    ws = pkg.alloc_workspace(w.T, w.N, w.H, w.d, w.d, w.M, dev)
    pkg.gdp_prefill_varlen(_args(w, d, ro, rf, rc, ws))
    torch.cuda.synchronize()
    del ws

    lib = pkg.load_library()
    no_ws = torch.empty(0, dtype=torch.uint8, device=dev)  # ignored by the static-scratch entry point
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):  # two calls in a row share the static scratch
        o, f, c = outputs()
        a = _args(w, d, o, f, c, no_ws)
        st = lib.gdp_prefill_varlen_static_scratch(ctypes.byref(a), ctypes.c_void_p(stream))
        assert st == pkg.GDP_OK, pkg.gdp_last_error()
        torch.cuda.synchronize()
        assert torch.equal(o, ro), f"call {call}: output differs from the caller-workspace call"
        assert torch.equal(f, rf), f"call {call}: final state differs from the caller-workspace call"
        assert torch.equal(c, rc), f"call {call}: chunk states differ from the caller-workspace call"
    ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale,
                         initial_state=w.initial_state, chunk_states=True)
    check_o(o.cpu(), ref["o"], label="o (static scratch) vs oracle")
    check_state(f.cpu(), ref["final_state"], label="final state (static scratch) vs oracle")
    check_state(c[:w.NT].cpu(), ref["chunk_states"], label="chunk states (static scratch) vs oracle", seq_offsets=ref["chunk_offsets"])


def test_static_scratch_rejects_oversized_shape(cuda_device):
    T, N, H, d, M = 65536, 1, 32, 128, 2
    assert pkg.gdp_prefill_workspace_bytes(T, N, H, d, d, M) > pkg.gdp_static_scratch_bytes()
    a = pkg.GdpPrefillArgs()
    a.T, a.N, a.H, a.K, a.V, a.num_householder = T, N, H, d, d, M
    lib = pkg.load_library()
    st = lib.gdp_prefill_varlen_static_scratch(ctypes.byref(a), None)
    assert st == pkg.GDP_ERR_WORKSPACE
    assert "static scratch" in pkg.gdp_last_error()
