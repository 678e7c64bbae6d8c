"""GPU parity: the CUDA path through the C ABI against the float64 oracle.

Small cases are compared element by element on every output; the full-size
workloads are compared on sampled heads (every token, every chunk state and
the final state of those heads) in the launch configuration the bench times.
Descriptors and untouched cache slots are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom, make_workload
from tests._parity import check_o, check_state
from tests.gpu_helpers import run, to_dev

pytestmark = pytest.mark.gpu


def _oracle(w, heads=None, **kw):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, state=w.state, state_indices=w.state_indices,
                          chunk_states=w.return_chunk_states, heads=heads, **kw)


def _compare(w, o, fin, cs, ref, heads=None):
    check_o(o.cpu(), ref["o"], heads=heads, cu_seqlens=w.cu_seqlens)
    if fin is not None and ref["final_state"] is not None:
        check_state(fin.cpu(), ref["final_state"], heads=heads, label="final_state")
    if cs is not None:
        nt = ref["chunk_states"].shape[0]
        assert nt == w.NT
        check_state(cs[:nt].cpu(), ref["chunk_states"], heads=heads, label="chunk_states", seq_offsets=ref["chunk_offsets"])
        if cs.shape[0] > nt:  # rows past the real count are not written
            assert torch.count_nonzero(cs[nt:]).item() == 0


# ---------------------------------------------------------------- descriptors (bit-exact)

@pytest.mark.parametrize("lengths,M", [([100, 257, 64, 1000], 2), ([257], 3), ([64, 0, 65, 1], 1),
                                       ([1] * 37 + [4000], 4), (list(range(0, 3000, 7)), 3), ([0, 0], 2),
                                       ([5] * 3000, 2)])
@pytest.mark.parametrize("cu_dtype", [torch.int32, torch.int64])
def test_descriptors_bit_exact(cuda_device, lengths, M, cu_dtype):
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=cu_dtype)
    T, N = int(cu[-1]), len(lengths)
    ci, cid, co = pkg.gdp_build_descriptors(cu.to(cuda_device), T, M)
    rci, rcid, rco, _ = oracle.descriptors(cu.numpy(), M)
    np.testing.assert_array_equal(ci.cpu().numpy(), rci)
    np.testing.assert_array_equal(cid.cpu().numpy(), rcid)
    np.testing.assert_array_equal(co.cpu().numpy(), rco)
    assert ci.shape[0] == pkg.gdp_nt_pad(T, N) and cid.shape[0] == pkg.gdp_ntdp_pad(T, N, M)


# ---------------------------------------------------------------- the five workloads

def test_workload1_gdn_tiny(cuda_device):
    w = make_workload(1)
    o, fin, cs, _ = run(w, cuda_device)
    _compare(w, o, fin, cs, _oracle(w))


def test_workload2_varlen_chunk_states(cuda_device):
    w = make_workload(2)
    o, fin, cs, _ = run(w, cuda_device)
    _compare(w, o, fin, cs, _oracle(w))


def test_workload2_prebuilt_descriptors(cuda_device):
    w = make_workload(2)
    a = run(w, cuda_device)
    b = run(w, cuda_device, prebuilt=True)
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)


@pytest.mark.slow
def test_workload3_l2norm_batch(cuda_device):
    w = make_workload(3)
    heads = [0, 5, 10, 15]
    o, fin, cs, _ = run(w, cuda_device)
    _compare(w, o, fin, cs, _oracle(w, heads=heads), heads=heads)


@pytest.mark.slow
def test_workload4_long_context(cuda_device):
    w = make_workload(4)
    heads = [0, 31]
    o, fin, cs, d = run(w, cuda_device)
    o, fin, cs = o[:, heads].cpu(), fin[:, heads].cpu(), cs[:, heads].cpu()
    del d
    torch.cuda.empty_cache()
    ref = _oracle(w, heads=heads)
    check_o(o, ref["o"][:, heads])
    check_state(fin, ref["final_state"][:, heads], label="final_state")
    check_state(cs[:w.NT], ref["chunk_states"][:, heads], label="chunk_states", seq_offsets=ref["chunk_offsets"])


@pytest.mark.slow
def test_workload5_state_cache_graph(cuda_device):
    """Prebuilt descriptors, state cache in place, CUDA-graph capture and replay."""
    w = make_workload(5)
    heads = [0, 7, 15]
    d = to_dev(w, cuda_device)
    pristine = d["state"].clone()
    ci, cid, co = pkg.gdp_build_descriptors(d["cu"], w.T, w.M)
    out = torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=cuda_device)
    ws = pkg.alloc_workspace(w.T, w.N, w.H, w.d, w.d, w.M, cuda_device)
    args = pkg.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale, None, d["state"],
                         d["sidx"], out, None, None, ci, cid, co, None, None, False, ws, None)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.capture_begin()
        pkg.gdp_prefill_varlen(args, s.cuda_stream)
        g.capture_end()
    torch.cuda.synchronize()
    assert torch.equal(d["state"], pristine)  # capture runs nothing
    g.replay()
    torch.cuda.synchronize()
    o_graph, cache_graph = out.clone(), d["state"].clone()
    ref = _oracle(w, heads=heads)
    check_o(o_graph.cpu(), ref["o"], heads=heads)
    sidx = w.state_indices.tolist()
    used = [s_ for s_ in sidx if s_ >= 0]
    unused = [s_ for s_ in range(w.state.shape[0]) if s_ not in used]
    cache_cpu = cache_graph.cpu()
    assert torch.equal(cache_cpu[unused], w.state[unused])  # untouched slots bit-identical
    check_state(cache_cpu[used][:, heads], ref["state_out"][used][:, heads], label="cache slots")
    # an eager run on the pristine cache gives the same bits as the replay
    d["state"].copy_(pristine)
    pkg.gdp_prefill_varlen(args)
    torch.cuda.synchronize()
    assert torch.equal(out, o_graph) and torch.equal(d["state"], cache_graph)


# ------------------------------------------- segmented mode (few chains, long sequences)

def test_segmented_uneven_lengths(cuda_device):
    """Chunk segments with the state carried between them; sequences ending in different
    segments (the shapes qualify: 12 chains, > 3 x 128 expanded chunks)."""
    w = make_custom([12345, 5000, 30], 4, 128, 2, seed=71, init_sigma=0.1, chunk_states=True)
    heads = [0, 3]
    o, fin, cs, _ = run(w, cuda_device)
    ref = _oracle(w, heads=heads)
    check_o(o.cpu(), ref["o"], heads=heads)
    check_state(fin.cpu(), ref["final_state"], heads=heads, label="final_state")
    check_state(cs[:w.NT].cpu(), ref["chunk_states"], heads=heads, label="chunk_states", seq_offsets=ref["chunk_offsets"])


def test_segmented_cache_graph(cuda_device):
    """Segmented mode inside a CUDA graph (internal streams fork from and join the capturing
    stream) with the state cache, against the oracle and against an eager call."""
    w = make_custom([12000, 700], 2, 128, 2, seed=72, cache_slots=4, cache_sigma=0.1, padding_slots=1)
    d = to_dev(w, cuda_device)
    pristine = d["state"].clone()
    out = torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=cuda_device)
    ws = pkg.alloc_workspace(w.T, w.N, w.H, w.d, w.d, w.M, cuda_device)
    args = pkg.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale, None, d["state"],
                         d["sidx"], out, None, None, None, None, None, None, None, False, ws, None)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g.capture_begin()
        pkg.gdp_prefill_varlen(args, s.cuda_stream)
        g.capture_end()
    torch.cuda.synchronize()
    assert torch.equal(d["state"], pristine)
    g.replay()
    torch.cuda.synchronize()
    o_graph, cache_graph = out.clone(), d["state"].clone()
    ref = _oracle(w)
    check_o(o_graph.cpu(), ref["o"])
    used = [s_ for s_ in w.state_indices.tolist() if s_ >= 0]
    check_state(cache_graph.cpu()[used], ref["state_out"][used], label="cache slots")
    d["state"].copy_(pristine)
    pkg.gdp_prefill_varlen(args)
    torch.cuda.synchronize()
    assert torch.equal(out, o_graph) and torch.equal(d["state"], cache_graph)


# ---------------------------------------------------------------- edge cases

EDGE = {
    "single_token": dict(lengths=[1], H=1, d=64, M=1),
    "ragged_tails_m3": dict(lengths=[63, 64, 65, 21, 22, 43], H=2, d=128, M=3, init_sigma=0.2, chunk_states=True),
    "chunk_aligned_m2": dict(lengths=[128, 64], H=2, d=128, M=2, init_sigma=0.2, chunk_states=True),
    "m4_d64": dict(lengths=[130, 5], H=3, d=64, M=4, init_sigma=0.1, chunk_states=True),
    "m8": dict(lengths=[40, 9], H=2, d=128, M=8, init_sigma=0.1),
    "empty_sequences": dict(lengths=[0, 17, 0, 0, 70, 0], H=2, d=128, M=2, init_sigma=0.3, chunk_states=True),
    "l2norm_m1": dict(lengths=[300], H=2, d=128, M=1, normalised=False, use_qk_l2norm=True),
    "strong_decay": dict(lengths=[200], H=2, d=128, M=2, decay=8.0, init_sigma=0.3),
    # chunk decays around 2^-20: a mix of chunks whose state decay is deferred and chunks
    # whose decay is applied to the state at once, with chunk states requested
    "mixed_decay": dict(lengths=[700, 333], H=2, d=128, M=2, decay=0.9, init_sigma=0.2, chunk_states=True),
    # chunk decays ~2^-9: the deferred decay product is renormalised every few chunks
    "frequent_renorm": dict(lengths=[900], H=2, d=128, M=3, decay=0.6, init_sigma=0.2, chunk_states=True),
    "no_gates": dict(lengths=[90, 33], H=2, d=64, M=2, with_g=False, with_beta=False, init_sigma=0.1),
    "many_short": dict(lengths=[3] * 50 + [1] * 20, H=2, d=128, M=3, chunk_states=True, init_sigma=0.1),
}


@pytest.mark.parametrize("name", sorted(EDGE))
def test_edge_cases(cuda_device, name):
    w = make_custom(seed=sorted(EDGE).index(name) + 500, name=name, **EDGE[name])
    o, fin, cs, _ = run(w, cuda_device)
    _compare(w, o, fin, cs, _oracle(w))


def test_all_empty_batch(cuda_device):
    w = make_custom([0, 0, 0], 2, 64, 2, init_sigma=0.5)
    o, fin, cs, _ = run(w, cuda_device)
    assert o.numel() == 0
    assert torch.equal(fin.cpu(), w.initial_state)


def test_int64_cu_seqlens_and_default_scale(cuda_device):
    w = make_custom([70, 130], 2, 128, 2, seed=3, init_sigma=0.1)
    d = to_dev(w, cuda_device, cu_dtype=torch.int64)
    o, fin, _, _ = run(w, cuda_device, d=d, scale=0.0)  # 0.0 selects 1/sqrt(K)
    _compare(w, o, fin, None, _oracle(w))


def test_strided_inputs(cuda_device):
    """Inputs that are views into wider buffers (head and row strides honoured)."""
    w = make_custom([50, 77], 3, 128, 2, seed=8, init_sigma=0.1)
    d = to_dev(w, cuda_device)
    for key in ("q", "k", "v"):
        t = d[key]
        wide = torch.zeros(t.shape[0], t.shape[1] + 1, t.shape[2] + 16, dtype=t.dtype, device=t.device)
        wide[:, 1:, 8:8 + t.shape[2]] = t
        d[key] = wide[:, 1:, 8:8 + t.shape[2]]
        assert not d[key].is_contiguous()
    o, fin, _, _ = run(w, cuda_device, d=d)
    _compare(w, o, fin, None, _oracle(w))


def test_resume_from_final_state(cuda_device):
    """Final-state chaining on the GPU: a sequence split at a non-aligned token and resumed."""
    w = make_custom([100, 150], 2, 128, 2, seed=21, init_sigma=0.2)
    d = to_dev(w, cuda_device)
    q, k, v, g, beta = d["q"], d["k"], d["v"], d["g"], d["beta"]
    s0, s1, cut = 100, 250, 170

    def part(a, b, init):
        cu = torch.tensor([0, b - a], dtype=torch.int32, device=cuda_device)
        return pkg.chunk_gated_delta_product(q[a:b], k[2 * a:2 * b], v[2 * a:2 * b], g[a:b], beta[2 * a:2 * b], cu,
                                             2, w.scale, initial_state=init, output_final_state=True)

    o1, f1 = part(s0, cut, d["init"][1:2].contiguous())
    o2, f2 = part(cut, s1, f1)
    torch.cuda.synchronize()
    ref = _oracle(w)
    check_o(torch.cat([o1, o2]).cpu(), ref["o"][s0:s1])
    check_state(f2.cpu(), ref["final_state"][1:2], label="resumed final")


def test_deterministic(cuda_device):
    w = make_custom([300, 45], 4, 128, 3, seed=4, init_sigma=0.1, chunk_states=True)
    a = run(w, cuda_device)
    b = run(w, cuda_device)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])


# ---------------------------------------------------------------- device-side error reporting

def test_bad_cu_seqlens_sets_status(cuda_device):
    """A decreasing cu_seqlens entry: status bit set, the bad sequence skipped, no fault."""
    w = make_custom([40, 40, 40], 2, 64, 2, seed=9)
    d = to_dev(w, cuda_device)
    d["cu"] = torch.tensor([0, 40, 30, 120], dtype=torch.int32, device=cuda_device)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    run(w, cuda_device, d=d, status=status)
    assert status.item() & pkg.GDP_DEV_ERR_CU_SEQLENS


def test_bad_slot_sets_status(cuda_device):
    w = make_custom([40, 40], 2, 64, 2, seed=10, cache_slots=4)
    d = to_dev(w, cuda_device)
    d["sidx"] = torch.tensor([1, 9], dtype=torch.int32, device=cuda_device)  # 9 >= num_slots
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    pristine = d["state"].clone()
    run(w, cuda_device, d=d, status=status)
    assert status.item() & pkg.GDP_DEV_ERR_SLOT
    assert torch.equal(d["state"][[0, 2, 3]], pristine[[0, 2, 3]])
