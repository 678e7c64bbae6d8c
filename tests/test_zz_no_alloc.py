"""gdp_prefill_varlen_static_scratch: the prefill for callers that cannot
allocate device memory (a plugin inside a runtime that owns all device memory,
or a host program that may not call cudaMalloc in its serving loop).

The entry point is called through the C ABI twice in a row on the same inputs
and each result is checked against the main entry point's result (which uses a
caller-owned workspace), within the parity tolerances of the other GPU tests.
A shape whose scratch need exceeds the static array is rejected before any
launch.  This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
from gdp_workloads import make_custom
from tests._parity import check_o, check_state

pytestmark = pytest.mark.gpu


def _args(w, d, out, fin, cs, workspace):
    return pkg.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale, d["init"], None, None,
                         out, fin, cs, None, None, None, None, None, w.use_qk_l2norm, workspace, None)


def test_static_scratch_matches_caller_workspace(cuda_device):
    w = make_custom([100, 257, 64, 300], 4, 128, 2, seed=77, init_sigma=0.1, chunk_states=True)
    assert pkg.gdp_prefill_workspace_bytes(w.T, w.N, w.H, w.d, w.d, w.M) <= pkg.GDP_STATIC_SCRATCH_BYTES
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

    lib = pkg.load_library()
    no_ws = torch.empty(0, dtype=torch.uint8, device=dev)  # ignored by the static-scratch entry point
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):  # two calls in a row share the static scratch
        o, f, c = outputs()
        a = _args(w, d, o, f, c, no_ws)
        st = lib.gdp_prefill_varlen_static_scratch(ctypes.byref(a), ctypes.c_void_p(stream))
        assert st == pkg.GDP_OK, pkg.gdp_last_error()
        torch.cuda.synchronize()
        check_o(o.cpu(), ro.cpu().double().numpy(), label="o (static scratch vs workspace)")
        check_state(f.cpu(), rf.cpu().double().numpy(), label="final state (static scratch vs workspace)")
        check_state(c[:w.NT].cpu(), rc[:w.NT].cpu().double().numpy(), label="chunk states (static scratch)")


def test_static_scratch_rejects_oversized_shape(cuda_device):
    T, N, H, d, M = 65536, 1, 32, 128, 2
    assert pkg.gdp_prefill_workspace_bytes(T, N, H, d, d, M) > pkg.GDP_STATIC_SCRATCH_BYTES
    a = pkg.GdpPrefillArgs()
    a.T, a.N, a.H, a.K, a.V, a.num_householder = T, N, H, d, d, M
    lib = pkg.load_library()
    st = lib.gdp_prefill_varlen_static_scratch(ctypes.byref(a), None)
    assert st == pkg.GDP_ERR_WORKSPACE
    assert "static scratch" in pkg.gdp_last_error()
