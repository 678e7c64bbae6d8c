"""Decode step (one token per sequence) against the float64 oracle and against the prefill.

The oracle's token loop with every sequence of length 1 is exactly the decode step
(Megatron-Core API page, parameters state / state_indices; FlashInfer API page, the
recurrence), so the same oracle serves: dense and state-cache modes, padding slots,
L2 norm, GDN (M = 1, d = 64) and M up to 4.  A prefill of L tokens followed by a
decode of token L+1 must equal a prefill of L+1 tokens.
"""
import ctypes

import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
from gdp_workloads import make_custom
from oracle import oracle
from tests._parity import check_o, check_state

pytestmark = pytest.mark.gpu


def _oracle(w):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, state=w.state, state_indices=w.state_indices)


@pytest.mark.parametrize("N,H,d,M,kw", [
    (64, 4, 128, 4, dict(cache_slots=96, cache_sigma=0.2, padding_slots=5)),
    (17, 3, 128, 2, dict(init_sigma=0.3)),
    (9, 2, 64, 1, dict(init_sigma=0.2)),
    (12, 2, 128, 3, dict(normalised=False, use_qk_l2norm=True, init_sigma=0.1)),
    (5, 2, 128, 2, dict()),
])
def test_decode_matches_oracle(cuda_device, N, H, d, M, kw):
    w = make_custom([1] * N, H, d, M, seed=300 + N, **kw)
    dev = cuda_device
    q, k, v, g, b = (t.to(dev) for t in (w.q, w.k, w.v, w.g, w.beta))
    ref = _oracle(w)
    if w.state is not None:
        cache = w.state.to(dev).clone()
        o = pkg.gated_delta_product_decode(q, k, v, g, b, M, w.scale, state=cache,
                                           state_indices=w.state_indices.to(dev))
        torch.cuda.synchronize()
        check_o(o.cpu(), ref["o"])
        used = [s for s in w.state_indices.tolist() if s >= 0]
        unused = [s for s in range(w.state.shape[0]) if s not in used]
        check_state(cache.cpu()[used], ref["state_out"][used], label="cache slots")
        assert torch.equal(cache.cpu()[unused], w.state[unused])
    else:
        init = None if w.initial_state is None else w.initial_state.to(dev)
        o, fin = pkg.gated_delta_product_decode(q, k, v, g, b, M, w.scale, initial_state=init,
                                                output_final_state=True, use_qk_l2norm_in_kernel=w.use_qk_l2norm)
        torch.cuda.synchronize()
        check_o(o.cpu(), ref["o"])
        check_state(fin.cpu(), ref["final_state"], label="final_state")


def test_decode_in_place_dense_state(cuda_device):
    """output_state == initial_state is an in-place update."""
    w = make_custom([1] * 8, 2, 128, 2, seed=331, init_sigma=0.3)
    dev = cuda_device
    s = w.initial_state.to(dev).clone()
    o, fin = pkg.gated_delta_product_decode(w.q.to(dev), w.k.to(dev), w.v.to(dev), w.g.to(dev), w.beta.to(dev), 2,
                                            w.scale, initial_state=s, output_final_state=True, output_state=s)
    torch.cuda.synchronize()
    ref = _oracle(w)
    check_o(o.cpu(), ref["o"])
    check_state(s.cpu(), ref["final_state"], label="in-place state")


def test_prefill_then_decode_equals_longer_prefill(cuda_device):
    """Prefill L tokens of each sequence, decode token L+1: same as a prefill of L+1 tokens."""
    lens = [40, 129, 7]
    M, H, d = 2, 2, 128
    w = make_custom([L + 1 for L in lens], H, d, M, seed=341, init_sigma=0.2)
    dev = cuda_device
    q, k, v, g, b = (t.to(dev) for t in (w.q, w.k, w.v, w.g, w.beta))
    cu = w.cu_seqlens.tolist()
    last = [cu[i + 1] - 1 for i in range(len(lens))]  # the decoded token of each sequence
    keep = [t for i in range(len(lens)) for t in range(cu[i], cu[i + 1] - 1)]
    kt = torch.tensor(keep, device=dev)
    kr = torch.tensor([t * M + j for t in keep for j in range(M)], device=dev)
    cu_short = torch.tensor([0] + list(torch.cumsum(torch.tensor(lens), 0)), dtype=torch.int32, device=dev)
    init = w.initial_state.to(dev)
    o_pre, s_pre = pkg.chunk_gated_delta_product(q[kt], k[kr], v[kr], g[kt], b[kr], cu_short, M, w.scale,
                                                 initial_state=init, output_final_state=True)
    lt = torch.tensor(last, device=dev)
    lr = torch.tensor([t * M + j for t in last for j in range(M)], device=dev)
    o_dec, s_dec = pkg.gated_delta_product_decode(q[lt], k[lr], v[lr], g[lt], b[lr], M, w.scale, initial_state=s_pre,
                                                  output_final_state=True)
    torch.cuda.synchronize()
    ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, w.scale, initial_state=w.initial_state)
    check_o(o_dec.cpu(), ref["o"][last], label="decoded token")
    check_state(s_dec.cpu(), ref["final_state"], label="state after decode")


def test_decode_rejects_bad_args(cuda_device):
    lib = pkg.load_library()
    w = make_custom([1] * 4, 2, 128, 2, seed=351)
    dev = cuda_device
    q, k, v = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    out = torch.empty((4, 2, 128), dtype=torch.bfloat16, device=dev)
    a = pkg.decode_args(q, k, v, None, None, 2, None, None, None, None, out, None, False, None)
    a.T = 5  # T != N
    assert lib.gdp_decode_step(ctypes.byref(a), None) == pkg.GDP_ERR_INVALID_ARG
    a.T = 4
    a.num_householder = 17
    assert lib.gdp_decode_step(ctypes.byref(a), None) == pkg.GDP_ERR_UNSUPPORTED
