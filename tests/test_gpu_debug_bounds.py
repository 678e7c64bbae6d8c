"""The debug-bounds build (libgdp_gb300_debug.so, -DGDP_DEBUG_BOUNDS=1) on the GPU.

Its kernels range-check every global index they derive from the descriptors, the sequence
table and the state-cache indices before the access; a failing check skips the access, sets
GDP_DEV_ERR_BOUNDS and records the first violation.  Checked here:
  * on valid calls of every plan (plain, split chains, segmented, state cache with prebuilt
    descriptors, decode) the debug build records nothing and matches the float64 oracle;
  * gdp_arm_bounds_test makes the next call check its output rows against T - 1: the (valid)
    stores of the last token's output fail their check, are skipped and recorded, and nothing
    else changes.  No access outside the caller's buffers is involved.
The debug library is swapped into the binding for these tests only.
"""
import contextlib

import pytest
import torch

import oracle
from chunked_gated_deltaproduct_gb300 import binding
from gdp_workloads import make_custom, make_workload
from tests._parity import check_o, check_state
from tests.gpu_helpers import run, to_dev

import chunked_gated_deltaproduct_gb300 as pkg

pytestmark = pytest.mark.gpu


@contextlib.contextmanager
def debug_library():
    from chunked_gated_deltaproduct_gb300 import build as libbuild

    libbuild.build(debug_bounds=True)
    saved = binding._lib
    binding._lib = binding.load_library(binding.DEBUG_LIB_PATH)
    try:
        pkg.gdp_debug_bounds_record()  # clear
        yield
    finally:
        binding._lib = saved


def _oracle(w):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, state=w.state, state_indices=w.state_indices,
                          chunk_states=w.return_chunk_states)


CASES = {
    "plain": lambda: make_custom([100, 257, 64, 1000, 3], 5, 128, 2, seed=41, init_sigma=0.1, chunk_states=True),
    "split_chains": lambda: make_workload(2),
    "segmented": lambda: make_custom([12288], 2, 128, 2, seed=43, init_sigma=0.05, chunk_states=True),
    "cache_prebuilt": lambda: make_custom([1, 77, 300, 5, 129], 3, 128, 4, seed=44, cache_slots=8, padding_slots=1,
                                          prebuilt_descriptors=True),
    "head64_m1": lambda: make_custom([65, 200], 2, 64, 1, seed=45, use_qk_l2norm=True, normalised=False),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_debug_build_records_nothing_on_valid_calls(cuda_device, name):
    w = CASES[name]()
    if name == "segmented":
        assert pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)["segments"] > 1
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    with debug_library():
        o, fin, cs, d = run(w, cuda_device, status=status, prebuilt=w.prebuilt_descriptors)
        rec = pkg.gdp_debug_bounds_record()
    assert rec["count"] == 0, rec
    assert int(status.item()) == 0
    ref = _oracle(w)
    check_o(o.cpu(), ref["o"], cu_seqlens=w.cu_seqlens)
    if w.state is not None:
        live = [int(s) for s in w.state_indices if s >= 0]
        check_state(d["state"][live].cpu(), ref["state_out"][live], label="cache slots")
    elif fin is not None:
        check_state(fin.cpu(), ref["final_state"], label="final_state")
    if cs is not None:
        nt = ref["chunk_states"].shape[0]
        check_state(cs[:nt].cpu(), ref["chunk_states"], label="chunk_states", seq_offsets=ref["chunk_offsets"])


def test_debug_build_decode_records_nothing(cuda_device):
    w = make_custom([1] * 9, 4, 128, 3, seed=46, cache_slots=16, padding_slots=2)
    d = to_dev(w, cuda_device)
    out = torch.empty((w.N, w.H, w.d), dtype=torch.bfloat16, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    with debug_library():
        args = pkg.decode_args(d["q"], d["k"], d["v"], d["g"], d["beta"], w.M, w.scale, None, d["state"], d["sidx"],
                               out, None, False, status)
        pkg.gdp_decode_step(args)
        torch.cuda.synchronize()
        rec = pkg.gdp_debug_bounds_record()
    assert rec["count"] == 0, rec
    assert int(status.item()) == 0
    ref = _oracle(w)
    check_o(out.cpu(), ref["o"])


def test_bounds_test_skips_and_records_the_last_rows(cuda_device):
    """The armed call's output rows are checked against T - 1: the last token's stores fail their
    check.  With an output buffer pre-filled with a sentinel, that row keeps the sentinel in every
    head, the record names the output site with index T - 1 and bound T - 1, and the rows of the
    earlier chunks match the oracle."""
    w = make_custom([300, 131], 2, 128, 2, seed=47, init_sigma=0.1)
    d = to_dev(w, cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    sentinel = torch.full((w.T, w.H, w.d), -7.0, dtype=torch.bfloat16, device=cuda_device)
    with debug_library():
        out = sentinel.clone()
        pkg.gdp_arm_bounds_test()
        res = pkg.chunk_gated_delta_product(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale,
                                            initial_state=d["init"], output_final_state=True, output=out,
                                            device_status=status)
        torch.cuda.synchronize()
        rec = pkg.gdp_debug_bounds_record()
        # the next call is unarmed: nothing recorded, every row written
        status2 = torch.zeros(1, dtype=torch.int32, device=cuda_device)
        out2 = sentinel.clone()
        pkg.chunk_gated_delta_product(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale,
                                      initial_state=d["init"], output_final_state=True, output=out2,
                                      device_status=status2)
        torch.cuda.synchronize()
        rec2 = pkg.gdp_debug_bounds_record()
    assert int(status.item()) == pkg.GDP_DEV_ERR_BOUNDS
    assert rec["count"] >= 1 and rec["site"] == "scan_out", rec
    assert rec["index"] == w.T - 1 and rec["bound"] == w.T - 1, rec
    assert torch.equal(out[w.T - 1], sentinel[w.T - 1])
    ref = _oracle(w)
    # the rows before the last sequence's last chunk are written and correct
    last_chunk_first_token = 300 + (131 * w.M - 1) // 64 * 64 // w.M
    check_o(out[:last_chunk_first_token].cpu(), ref["o"][:last_chunk_first_token])
    check_state(res[1].cpu(), ref["final_state"], label="final_state")
    assert int(status2.item()) == 0 and rec2["count"] == 0, rec2
    check_o(out2.cpu(), ref["o"])
