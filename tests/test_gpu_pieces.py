"""GPU parity of the split-chains form against the float64 oracle.

A call over few sequences and heads cuts every sequence into pieces of a few expanded
chunks: a first scan pass gives each piece's end state from a zero state (B) and from the
identity with V = 0 (Phi), a combine kernel chains the entering states
S_in(j + 1) = S_in(j) Phi_j + B_j, and a second pass runs every piece from its own.  Each
case below is split (checked through the plan query); its twin with 64 heads over the same
lengths runs the plain form, so both forms meet the same cases.
"""
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state
from tests.gpu_helpers import run, to_dev

pytestmark = pytest.mark.gpu

CASES = {
    "m2_chunk_states": dict(lengths=[100, 257, 64, 1000], H=2, d=128, M=2, init_sigma=0.1, chunk_states=True),
    "m3_straddle_l2norm": dict(lengths=[700, 33, 0, 410], H=2, d=64, M=3, normalised=False, use_qk_l2norm=True,
                               init_sigma=0.2, chunk_states=True),
    "m1_single_long": dict(lengths=[3000], H=1, d=128, M=1, init_sigma=0.1),
    "cache_with_padding": dict(lengths=[900, 120, 640], H=2, d=128, M=2, cache_slots=6, padding_slots=1),
    "bf16_state_f16_inputs": dict(lengths=[1500, 77], H=2, d=128, M=2, init_sigma=0.2,
                                  state_dtype=torch.bfloat16, qkv_dtype=torch.float16),
    "deferred_and_applied_decay": dict(lengths=[1200], H=2, d=128, M=3, decay=0.9, init_sigma=0.2,
                                       chunk_states=True),
    "no_gate_no_beta_m4": dict(lengths=[800, 300], H=2, d=64, M=4, with_g=False, with_beta=False,
                               init_sigma=0.1),
    "grouped_heads": dict(lengths=[1000, 260], H=4, d=64, M=2, hq=2, hk=2, hv=4, init_sigma=0.1,
                          chunk_states=True),
    # M does not divide the piece length: token-chunk starts fall at different local chunks per piece
    "m4_chunk_states_unaligned": dict(lengths=[900, 70], H=2, d=64, M=4, init_sigma=0.1, chunk_states=True),
    # both sequences are split, so the padded slot belongs to a split sequence
    "cache_padding_on_split": dict(lengths=[900, 700], H=2, d=128, M=2, cache_slots=4, padding_slots=1),
}
PLAIN_H = 64


def _oracle(w, heads=None):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                          initial_state=w.initial_state, state=w.state, state_indices=w.state_indices,
                          chunk_states=w.return_chunk_states, heads=heads)


def _check(w, o, fin, cs, d, heads=None):
    ref = _oracle(w, heads=heads)
    check_o(o.float().cpu(), ref["o"], heads=heads)
    if fin is not None and ref["final_state"] is not None:
        check_state(fin.cpu(), ref["final_state"], heads=heads, label="final_state")
    if cs is not None:
        check_state(cs[:w.NT].cpu(), ref["chunk_states"], heads=heads, label="chunk_states", seq_offsets=ref["chunk_offsets"])
    if w.state is not None:
        used = [s for s in w.state_indices.tolist() if s >= 0]
        unused = [s for s in range(w.state.shape[0]) if s not in used]
        cache = d["state"].cpu()
        assert torch.equal(cache[unused], w.state[unused])  # untouched slots bit-identical
        out = ref["state_out"][used]
        check_state(cache[used] if heads is None else cache[used][:, heads],
                    out if heads is None else out[:, heads], label="cache slots")


def _seed(name, plain):
    return 300 + 2 * sorted(CASES).index(name) + int(plain)


@pytest.mark.parametrize("name", sorted(CASES))
def test_split_chains_parity(cuda_device, name):
    kw = dict(CASES[name])
    w = make_custom(seed=_seed(name, False), **kw)
    plan = pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)
    assert plan["piece_chunks"] > 0 and plan["launches"] == 5, plan
    o, fin, cs, d = run(w, cuda_device)
    _check(w, o, fin, cs, d)


@pytest.mark.parametrize("name", sorted(CASES))
def test_plain_twin_parity(cuda_device, name):
    kw = dict(CASES[name])
    r = PLAIN_H // kw["H"]
    kw["H"] = PLAIN_H
    for key in ("hq", "hk", "hv"):  # keep the grouping ratios
        if key in kw:
            kw[key] *= r
    w = make_custom(seed=_seed(name, True), **kw)
    plan = pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)
    assert plan["piece_chunks"] == 0 and plan["segments"] == 1, plan
    heads = [0, PLAIN_H - 1]
    o, fin, cs, d = run(w, cuda_device)
    _check(w, o, fin, cs, d, heads=heads)


def test_split_chains_repeatable_and_graph_capturable(cuda_device):
    """Bit-identical results across eager calls and a CUDA-graph replay (state cache in place)."""
    w = make_custom([1100, 300, 5], 2, 128, 2, seed=331, cache_slots=5, cache_sigma=0.1, chunk_states=True)
    assert pkg.gdp_prefill_plan(w.T, w.N, w.H, w.d, w.d, w.M)["piece_chunks"] > 0
    d = to_dev(w, cuda_device)
    pristine = d["state"].clone()
    out = torch.empty((w.T, w.H, w.d), dtype=torch.bfloat16, device=cuda_device)
    cs = torch.zeros((pkg.gdp_nt_pad(w.T, w.N), w.H, w.d, w.d), dtype=torch.float32, device=cuda_device)
    ws = pkg.alloc_workspace(w.T, w.N, w.H, w.d, w.d, w.M, cuda_device)
    args = pkg.make_args(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu"], w.M, w.scale, None, d["state"],
                         d["sidx"], out, None, cs, None, None, None, None, None, False, ws, None)
    pkg.gdp_prefill_varlen(args)
    torch.cuda.synchronize()
    o1, c1, s1 = out.clone(), cs.clone(), d["state"].clone()
    d["state"].copy_(pristine)
    pkg.gdp_prefill_varlen(args)
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(cs, c1) and torch.equal(d["state"], s1)
    d["state"].copy_(pristine)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        g.capture_begin()
        pkg.gdp_prefill_varlen(args, s.cuda_stream)
        g.capture_end()
    torch.cuda.synchronize()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, o1) and torch.equal(cs, c1) and torch.equal(d["state"], s1)
    ref = _oracle(w)
    check_o(o1.float().cpu(), ref["o"])
    check_state(c1[:w.NT].cpu(), ref["chunk_states"], label="chunk_states", seq_offsets=ref["chunk_offsets"])
    used = [x for x in w.state_indices.tolist() if x >= 0]
    check_state(s1.cpu()[used], ref["state_out"][used], label="cache slots")
