"""Input variants against the float64 oracle (FlashInfer API page
"flashinfer.gdp_prefill.chunk_gated_delta_product", parameters q, k, v, g, beta,
initial_state): float16 q / k / v and output, q / k / v with fewer heads than the
state, the gate as alpha in linear space, bf16 / f16 g and beta, a bf16 initial
state -- through the prefill (one segment and the segmented mode) and the decode
step, at the tolerances of every other parity test.
"""
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state
from tests.gpu_helpers import run

pytestmark = pytest.mark.gpu

F16, BF16 = torch.float16, torch.bfloat16


def _oracle(w):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, state=w.state, state_indices=w.state_indices,
                          chunk_states=w.return_chunk_states, g_is_alpha=w.g_is_alpha)


def _check_prefill(w, dev):
    o, fin, cs, _ = run(w, dev)
    assert o.dtype == w.q.dtype and tuple(o.shape) == (w.T, w.H, w.d)
    ref = _oracle(w)
    check_o(o.cpu(), ref["o"])
    if fin is not None:
        assert fin.dtype == torch.float32
        check_state(fin.cpu(), ref["final_state"], label="final_state")
    if cs is not None:
        nt = ref["chunk_states"].shape[0]
        check_state(cs[:nt].cpu(), ref["chunk_states"], label="chunk_states", seq_offsets=ref["chunk_offsets"])
    return ref


VARLEN = dict(lengths=[100, 257, 64, 1000], H=8, d=128, M=2, decay=0.05, init_sigma=0.1, chunk_states=True)

CASES = {
    # float16 q / k / v (and output)
    "f16_varlen_chunk_states": dict(VARLEN, qkv_dtype=F16),
    "f16_l2norm_m3_d64": dict(lengths=[300, 65, 1], H=4, d=64, M=3, normalised=False, use_qk_l2norm=True,
                              qkv_dtype=F16),
    # chunk decay about 2^-14: images divided by it (T factors up to 2^14 before the f16 scaling)
    "f16_fast_images_large_shift": dict(lengths=[700, 90], H=2, d=128, M=2, decay=0.6, init_sigma=0.3,
                                        qkv_dtype=F16),
    "f16_slow_images": dict(lengths=[700], H=2, d=128, M=2, decay=3.0, init_sigma=0.3, qkv_dtype=F16),
    # grouped heads: H = max(Hq, Hv) state heads
    "gva_q2_k2_v8": dict(VARLEN, hq=2, hk=2, hv=8),
    "gqa_q8_k2_v2": dict(lengths=[130, 600], H=8, d=128, M=2, hq=8, hk=2, hv=2),
    "k_follows_q_v_shared": dict(lengths=[130, 600], H=4, d=64, M=3, hq=4, hk=4, hv=1),
    # linear-space alpha gate, natural-log gate in 16-bit types
    "alpha_f32": dict(VARLEN, g_is_alpha=True),
    "alpha_bf16": dict(lengths=[500, 33], H=4, d=128, M=2, g_is_alpha=True, g_dtype=BF16),
    "alpha_f16_strong_decay": dict(lengths=[500], H=2, d=128, M=4, decay=2.0, g_is_alpha=True, g_dtype=F16,
                                   init_sigma=0.5),
    "g_bf16": dict(lengths=[300, 77], H=4, d=128, M=2, g_dtype=BF16),
    "g_f16": dict(lengths=[300, 77], H=4, d=128, M=2, g_dtype=F16),
    # beta in the q/k/v type
    "beta_bf16": dict(lengths=[300, 77], H=4, d=128, M=2, beta_dtype=BF16),
    "beta_f16_with_f16_inputs": dict(lengths=[300, 77], H=4, d=128, M=2, qkv_dtype=F16, beta_dtype=F16),
    # bf16 initial state
    "init_bf16": dict(VARLEN, state_dtype=BF16),
    # all at once
    "all_variants": dict(lengths=[40, 300, 129], H=8, d=128, M=3, normalised=False, use_qk_l2norm=True,
                         qkv_dtype=F16, hq=4, hk=4, hv=8, g_is_alpha=True, g_dtype=F16, beta_dtype=F16,
                         init_sigma=0.2, state_dtype=BF16, chunk_states=True),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_variant(cuda_device, name):
    kw = dict(CASES[name])
    w = make_custom(kw.pop("lengths"), kw.pop("H"), kw.pop("d"), kw.pop("M"), seed=700 + len(name), name=name, **kw)
    _check_prefill(w, cuda_device)


def test_alpha_zero_resets_state(cuda_device):
    """alpha = 0 (the edge of the page's range (0, 1]) wipes the state; the kernel's floor of
    exp(-80) leaves a remainder far below the tolerance."""
    w = make_custom([200, 90], 4, 128, 2, seed=731, g_is_alpha=True, init_sigma=1.0, chunk_states=True)
    w.g[[5, 64, 130, 131, 250]] = 0.0
    _check_prefill(w, cuda_device)


def test_segmented_f16_grouped(cuda_device):
    """The segmented mode (one long sequence, few chains) with float16 inputs and grouped heads."""
    w = make_custom([12800], 2, 128, 2, seed=741, decay=0.05, init_sigma=0.1, chunk_states=True, qkv_dtype=F16,
                    hq=1, hk=1, hv=2, g_is_alpha=True, beta_dtype=F16)
    _check_prefill(w, cuda_device)


DECODE = {
    "f16": dict(qkv_dtype=F16, init_sigma=0.3),
    "gva": dict(hq=1, hk=1, hv=4, init_sigma=0.3),
    "gqa": dict(hq=4, hk=2, hv=2, init_sigma=0.3),
    "alpha_bf16_beta_bf16": dict(g_is_alpha=True, g_dtype=BF16, beta_dtype=BF16, init_sigma=0.3),
    "init_bf16_l2norm": dict(state_dtype=BF16, init_sigma=0.3, normalised=False, use_qk_l2norm=True),
    "f16_cache": dict(qkv_dtype=F16, beta_dtype=F16, g_dtype=F16, cache_slots=40, cache_sigma=0.2, padding_slots=3),
}


@pytest.mark.parametrize("name", sorted(DECODE))
def test_decode_variant(cuda_device, name):
    w = make_custom([1] * 24, 4, 128, 3, seed=760 + len(name), **DECODE[name])
    dev = cuda_device
    q, k, v, g, b = (t.to(dev) for t in (w.q, w.k, w.v, w.g, w.beta))
    ref = _oracle(w)
    if w.state is not None:
        cache = w.state.to(dev).clone()
        o = pkg.gated_delta_product_decode(q, k, v, g, b, 3, w.scale, state=cache,
                                           state_indices=w.state_indices.to(dev), g_is_alpha=w.g_is_alpha,
                                           use_qk_l2norm_in_kernel=w.use_qk_l2norm)
        torch.cuda.synchronize()
        used = [s for s in w.state_indices.tolist() if s >= 0]
        check_state(cache.cpu()[used], ref["state_out"][used], label="cache slots")
    else:
        init = None if w.initial_state is None else w.initial_state.to(dev)
        o, fin = pkg.gated_delta_product_decode(q, k, v, g, b, 3, w.scale, initial_state=init,
                                                output_final_state=True, use_qk_l2norm_in_kernel=w.use_qk_l2norm,
                                                g_is_alpha=w.g_is_alpha)
        torch.cuda.synchronize()
        check_state(fin.cpu(), ref["final_state"], label="final_state")
    assert o.dtype == w.q.dtype
    check_o(o.cpu(), ref["o"])
