"""Host-side canaries around the buffers a call writes.

Every output buffer (o, the final state, the chunk states) and the workspace is
carved out of a larger allocation whose guard bands before and after it hold a
fixed byte pattern; after the call the bands must be unchanged, so no kernel
writes outside the buffers it was given.  Each way a call runs (gdp_prefill_varlen plain,
split or segmented; gdp_prefill_varlen_fused whole or split into pieces) is covered, and
the outputs are checked against the oracle as well.
"""
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state

pytestmark = pytest.mark.gpu

GUARD = 64 << 10  # bytes of each band (keeps 256-byte alignment of the carved buffer)
PATTERN = 0xA5


class Guarded:
    """A buffer of `nbytes` between two guard bands of PATTERN bytes."""

    def __init__(self, nbytes, dev):
        self.n = nbytes
        self.raw = torch.full((GUARD + nbytes + GUARD,), PATTERN, dtype=torch.uint8, device=dev)

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def bands_intact(self):
        lo, hi = self.raw[:GUARD], self.raw[GUARD + self.n:]
        return bool((lo == PATTERN).all()) and bool((hi == PATTERN).all())


@pytest.mark.parametrize("lengths,H,d,M,kind", [
    ([5 * i + 3 for i in range(40)], 2, 128, 3, "staged"),
    ([100, 257, 64, 300], 4, 128, 2, "staged split"),
    ([12288], 1, 128, 2, "staged segmented"),
    ([5 * i + 3 for i in range(40)], 2, 128, 3, "fused"),
    ([100, 257, 64, 300], 4, 128, 2, "fused split"),
])
def test_no_write_outside_the_given_buffers(cuda_device, lengths, H, d, M, kind):
    dev = cuda_device
    w = make_custom(lengths, H, d, M, seed=123, init_sigma=0.1, chunk_states=True)
    fused = kind.startswith("fused")
    plan = pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M) if fused else pkg.gdp_prefill_plan(
        w.T, w.N, w.H, w.d, w.d, w.M)
    got = ("fused" if fused else "staged") + (" segmented" if plan.get("segments", 1) > 1 else
                                              " split" if plan["piece_chunks"] else "")
    assert kind == got
    nt = pkg.gdp_nt_pad(w.T, w.N)
    g_out = Guarded(w.T * w.H * w.d * 2, dev)
    g_fin = Guarded(w.N * w.H * w.d * w.d * 4, dev)
    g_cs = Guarded(nt * w.H * w.d * w.d * 4, dev)
    g_ws = Guarded(pkg.gdp_prefill_workspace_bytes(w.T, w.N, w.H, w.d, w.d, w.M), dev)
    out = g_out.view(torch.bfloat16, (w.T, w.H, w.d))
    fin = g_fin.view(torch.float32, (w.N, w.H, w.d, w.d))
    cs = g_cs.view(torch.float32, (nt, w.H, w.d, w.d))
    cs.zero_()
    ws = g_ws.view(torch.uint8, (g_ws.n,))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    q, k, v, g, beta, cu, init = (t.to(dev) for t in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.initial_state))
    a = pkg.make_args(q, k, v, g, beta, cu, w.M, w.scale, init, None, None, out, fin, cs, None, None, None, None,
                      None, False, ws, status)
    (pkg.gdp_prefill_varlen_fused if fused else pkg.gdp_prefill_varlen)(a)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for name, gb in (("output", g_out), ("final state", g_fin), ("chunk states", g_cs), ("workspace", g_ws)):
        assert gb.bands_intact(), f"a kernel wrote outside the {name} buffer"
    assert torch.count_nonzero(cs[w.NT:]).item() == 0  # rows past the real count stay untouched
    ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, initial_state=w.initial_state,
                         chunk_states=True)
    check_o(out.cpu(), ref["o"], cu_seqlens=w.cu_seqlens)
    check_state(fin.cpu(), ref["final_state"], label="final_state")
    check_state(cs[:w.NT].cpu(), ref["chunk_states"], label="chunk_states", seq_offsets=ref["chunk_offsets"])
