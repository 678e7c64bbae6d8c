"""Failure detection on the GPU without a GPU fault: the bounded waits.

Every spin-wait of the kernels is bounded.  gdp_arm_wait_expiry_test arms one
call so that its waits give up after a few milliseconds and the CTA of sequence
0, head 0 (of the fused kernel, or of the staged scan) withholds its first copy: one wait runs out (a
flag that nothing sets), the CTA drains its own tensor-core work and copies,
frees its tensor memory and returns.  The test checks that the call completes
promptly, that the status word carries GDP_DEV_ERR_TIMEOUT, and that the
context stays usable: the next call on the same inputs matches the oracle.
No test here faults, traps or hangs the GPU.
"""
import time

import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state
from tests.gpu_helpers import run, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fused", [False, True])
def test_wait_expiry_sets_timeout_and_context_survives(cuda_device, fused):
    """The staged scan (gdp_prefill_varlen) and the fused kernel (gdp_prefill_varlen_fused) each
    withhold one copy."""
    w = make_custom([100, 37], 2, 128, 2, seed=31, init_sigma=0.1)
    plan = pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M) if fused else pkg.gdp_prefill_plan(
        w.T, w.N, w.H, w.d, w.d, w.M)
    assert plan["piece_chunks"] == 0  # one launch of the kernel under test
    d = to_dev(w, cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pkg.gdp_arm_wait_expiry_test(2_000_000)  # 2 ms
    t0 = time.perf_counter()
    run(w, cuda_device, d=d, status=status, fused=fused)  # synchronises
    took = time.perf_counter() - t0
    st = int(status.item())
    assert st & pkg.GDP_DEV_ERR_TIMEOUT, f"status {st:#x}: the withheld copy's wait did not run out"
    assert st & ~pkg.GDP_DEV_ERR_TIMEOUT == 0, f"status {st:#x}"
    assert took < 5.0, f"the expired call took {took:.2f} s"
    # the context is usable and the next (unarmed) call is correct
    status.zero_()
    o, fin, _, _ = run(w, cuda_device, d=d, status=status, fused=fused)
    assert int(status.item()) == 0
    ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, initial_state=w.initial_state)
    check_o(o.cpu(), ref["o"])
    check_state(fin.cpu(), ref["final_state"], label="final_state")


def test_arm_rejects_out_of_range_limit():
    for bad in (0, 10, 2_000_000_000):
        with pytest.raises(pkg.GdpError):
            pkg.gdp_arm_wait_expiry_test(bad)
