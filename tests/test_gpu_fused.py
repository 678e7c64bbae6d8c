"""GPU parity of the fused prefill kernel (WY work, state scan, outputs and state scatter in one
CTA per (sequence, head)) against the float64 oracle.

Every case runs through gdp_prefill_varlen_fused (the plan of gdp_prefill_fused), so these
tests hold the fused kernel itself to the parity bar: per-head relative L2 <= 5e-3 on o and
<= 2e-3 on final and chunk states (and per (sequence, head) on states), max |delta o| <= 2e-2,
untouched cache slots bit for bit.  The cases cover ragged chunk tails, empty and one-token
sequences, chunks whose decay falls below 2^-20 (applied to the state between the two scan
products) and long chains that cross many renormalisations, the state cache with padding
slots, in-kernel L2 normalisation, grouped heads and M = 2 .. 8.
"""
import numpy as np
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state
from tests.gpu_helpers import run

pytestmark = pytest.mark.gpu

CASES = {
    "m2_ragged": dict(lengths=[100, 257, 64, 1000, 37, 0, 1, 5] + [33] * 25, H=2, M=2, init_sigma=0.1,
                      chunk_states=True),
    "m3_straddle": dict(lengths=[63, 64, 65, 21, 22, 43] * 6, H=2, M=3, init_sigma=0.2, chunk_states=True),
    "m4_serving": dict(lengths=[16, 700, 91, 2048, 1, 0, 300] * 5 + [50], H=2, M=4, init_sigma=0.1),
    "m8": dict(lengths=[130, 7, 64] * 11, H=1, M=8, init_sigma=0.1, chunk_states=True),
    "l2norm_m3": dict(lengths=[500, 129, 3] * 11, H=2, M=3, normalised=False, use_qk_l2norm=True),
    "strong_decay": dict(lengths=[200, 64, 65] * 11, H=2, M=2, decay=8.0, init_sigma=0.3, chunk_states=True),
    "mixed_decay": dict(lengths=[700, 333] * 17, H=1, M=2, decay=0.9, init_sigma=0.2, chunk_states=True),
    "frequent_renorm": dict(lengths=[2000, 900] * 17, H=1, M=3, decay=0.6, init_sigma=0.2, chunk_states=True),
    "no_gates": dict(lengths=[90, 33, 64] * 11, H=2, M=2, with_g=False, with_beta=False, init_sigma=0.1),
    "zero_state_chunks": dict(lengths=[128, 129, 1] * 11, H=2, M=2, chunk_states=True),
    "long_chain": dict(lengths=[20000], H=2, M=2, decay=0.02, init_sigma=0.05, chunk_states=True),
    # few chains: the fused kernel splits them into pieces (pass 1, combine, pass 2)
    "split_varlen": dict(lengths=[100, 257, 64, 1000], H=8, M=2, decay=0.05, init_sigma=0.1, chunk_states=True),
    "split_long_m3": dict(lengths=[8192, 5], H=4, M=3, decay=0.02, init_sigma=0.05, chunk_states=True),
    "split_strong_decay": dict(lengths=[3000, 70], H=2, M=2, decay=2.0, init_sigma=0.3, chunk_states=True),
}
SPLIT = {"long_chain", "split_varlen", "split_long_m3", "split_strong_decay"}


def _oracle(w):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, state=w.state, state_indices=w.state_indices,
                          chunk_states=w.return_chunk_states)


def _check(w, o, fin, cs, ref):
    check_o(o.cpu(), ref["o"], cu_seqlens=w.cu_seqlens)
    if fin is not None and ref["final_state"] is not None:
        check_state(fin.cpu(), ref["final_state"], label="final_state")
    if cs is not None:
        nt = ref["chunk_states"].shape[0]
        check_state(cs[:nt].cpu(), ref["chunk_states"], label="chunk_states", seq_offsets=ref["chunk_offsets"])
        if cs.shape[0] > nt:
            assert torch.count_nonzero(cs[nt:]).item() == 0


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_parity(cuda_device, name):
    w = make_custom(seed=sorted(CASES).index(name) + 900, d=128, name=name, **CASES[name])
    plan = pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M)
    assert plan is not None, "the fused kernel should serve this shape"
    assert (plan["piece_chunks"] > 0) == (name in SPLIT)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    o, fin, cs, _ = run(w, cuda_device, status=status, fused=True)
    assert int(status.item()) == 0
    _check(w, o, fin, cs, _oracle(w))


def test_fused_state_cache_in_place(cuda_device):
    """Cache mode: slots read and written in place, -1 padding sequences start from zero and
    write nothing, untouched slots bit-identical."""
    w = make_custom([100, 0, 513, 64, 1, 300] * 6, 2, 128, 4, seed=77, cache_slots=48, cache_sigma=0.1,
                    padding_slots=5)
    assert pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M) is not None
    o, fin, cs, d = run(w, cuda_device, fused=True)
    ref = _oracle(w)
    check_o(o.cpu(), ref["o"], cu_seqlens=w.cu_seqlens)
    cache = d["state"].cpu()
    used = set(int(s) for s in w.state_indices.tolist() if s >= 0)
    for s in range(w.state.shape[0]):
        if s not in used:
            assert torch.equal(cache[s], w.state[s]), f"slot {s} was touched"
    check_state(cache[sorted(used)], ref["state_out"][sorted(used)], label="cache slots")


def test_fused_split_state_cache(cuda_device):
    """Split chains with the state cache: pieces read the slot through the combine kernel, the
    last piece writes it; padding sequences start from zero and write nothing."""
    w = make_custom([1500, 3, 700, 0], 4, 128, 2, seed=78, cache_slots=8, cache_sigma=0.1, padding_slots=1)
    assert pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M)["piece_chunks"] > 0
    o, fin, cs, d = run(w, cuda_device, fused=True)
    ref = _oracle(w)
    check_o(o.cpu(), ref["o"], cu_seqlens=w.cu_seqlens)
    cache = d["state"].cpu()
    used = set(int(s) for s in w.state_indices.tolist() if s >= 0)
    for s in range(w.state.shape[0]):
        if s not in used:
            assert torch.equal(cache[s], w.state[s]), f"slot {s} was touched"
    check_state(cache[sorted(used)], ref["state_out"][sorted(used)], label="cache slots")


def test_fused_longest_first_order(cuda_device):
    """Over whole sequences the fused kernel runs them longest first (a device-built order);
    lengths in rising order, equal lengths and an empty sequence come out right."""
    w = make_custom(list(range(1, 40)) + [0, 600, 600, 2000], 2, 128, 2, seed=79, init_sigma=0.1, chunk_states=True)
    assert pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M)["piece_chunks"] == 0
    o, fin, cs, _ = run(w, cuda_device, fused=True)
    _check(w, o, fin, cs, _oracle(w))


def test_fused_grouped_heads(cuda_device):
    """q, k with 2 heads serving 8 state heads (GVA): each input head feeds a run of state heads."""
    w = make_custom([300, 77, 1000] * 11, 8, 128, 2, seed=31, hq=2, hk=2, init_sigma=0.1, chunk_states=True)
    assert pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M) is not None
    o, fin, cs, _ = run(w, cuda_device, fused=True)
    _check(w, o, fin, cs, _oracle(w))


def test_fused_graph_replay_bit_identical(cuda_device):
    """The fused call captures into a CUDA graph; a replay gives the eager call's bits."""
    w = make_custom([500, 64, 3000] * 11, 2, 128, 2, seed=5, init_sigma=0.1, chunk_states=True)
    dev = cuda_device
    q, k, v, g, beta, cu, init = (t.to(dev) for t in (w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.initial_state))
    out = torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=dev)
    fin = torch.empty((w.N, w.H, w.d, w.d), dtype=torch.float32, device=dev)
    cs = torch.zeros((pkg.gdp_nt_pad(w.T, w.N), w.H, w.d, w.d), dtype=torch.float32, device=dev)
    ws = pkg.alloc_workspace(w.T, w.N, w.H, w.d, w.d, w.M, dev)
    a = pkg.make_args(q, k, v, g, beta, cu, w.M, w.scale, init, None, None, out, fin, cs, None, None, None, None, None,
                      False, ws, None)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        pkg.gdp_prefill_varlen_fused(a, s.cuda_stream)
    torch.cuda.synchronize()
    eager = (out.clone(), fin.clone(), cs.clone())
    out.zero_(), fin.zero_(), cs.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        graph.capture_begin()
        pkg.gdp_prefill_varlen_fused(a, s.cuda_stream)
        graph.capture_end()
    graph.replay()
    torch.cuda.synchronize()
    for x, y in zip((out, fin, cs), eager):
        assert torch.equal(x, y)


def test_fused_rejects_what_it_does_not_serve(cuda_device):
    """Another input type or head size is refused before any launch (the staged kernels serve it)."""
    w = make_custom([100, 37], 2, 64, 2, seed=3)
    assert pkg.gdp_prefill_fused(w.T, w.N, w.H, w.d, w.d, w.M) is None
    with pytest.raises(pkg.GdpError):
        run(w, cuda_device, fused=True)
    w16 = make_custom([100, 37], 2, 128, 2, seed=3, qkv_dtype=torch.float16)
    with pytest.raises(pkg.GdpError):
        run(w16, cuda_device, fused=True)
