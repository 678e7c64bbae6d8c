"""Pins of the float64 oracle against what the pages and the mathematics fix.

Each test states the fact it checks.  Together they are chosen so that a
dropped term, a wrong sign, a wrong row index (expanded vs token stream), a
decay applied per sub-row instead of per token, a transposed state or a
chunk-state row off by one fails at least one of them.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from gdp_workloads import make_custom
from tests._pins import f64, gdn_kmajor, rel_err, transition_bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _run(w, **kw):
    return oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale,
                          use_qk_l2norm=w.use_qk_l2norm, initial_state=w.initial_state,
                          state=w.state, state_indices=w.state_indices,
                          chunk_states=w.return_chunk_states, **kw)


def _read_kv(path):
    out = {}
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = [float(x) for x in vals]
    return out


def test_handworked_example():
    """Hand-worked n = 2 example (tests/golden/handworked_gdp_n2_d2.txt)."""
    f = _read_kv(os.path.join(GOLDEN, "handworked_gdp_n2_d2.txt"))
    bf = torch.bfloat16
    q = torch.tensor(f["q"]).reshape(2, 1, 2).to(bf)
    k = torch.tensor(f["k"]).reshape(4, 1, 2).to(bf)
    v = torch.tensor(f["v"]).reshape(4, 1, 2).to(bf)
    beta = torch.tensor(f["beta"], dtype=torch.float32).reshape(4, 1)
    g = torch.tensor(f["g"], dtype=torch.float32).reshape(2, 1)
    S0 = torch.tensor(f["S0"], dtype=torch.float32).reshape(1, 1, 2, 2)
    res = oracle.forward(q, k, v, g, beta, [0, 2], 2, f["scale"][0], initial_state=S0, chunk_states=True)
    np.testing.assert_allclose(res["o"].ravel(), f["o"], rtol=1e-6, atol=1e-7)
    np.testing.assert_allclose(res["final_state"].ravel(), f["final"], rtol=1e-6, atol=1e-7)
    np.testing.assert_array_equal(res["chunk_states"].ravel(), f["chunk0"])


@pytest.mark.parametrize("l2norm", [False, True])
def test_n1_is_gated_delta_rule(l2norm):
    """num_householder == 1 is the gated delta rule (FlashInfer page; GDN recurrence of the blog post)."""
    w = make_custom([5, 17, 70], 2, 8, 1, seed=11, normalised=not l2norm, use_qk_l2norm=l2norm,
                    decay=0.3, init_sigma=0.5)
    res = _run(w)
    o_ref, fin_ref = gdn_kmajor(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.scale,
                                S0_vmajor=w.initial_state, l2norm=l2norm)
    assert rel_err(res["o"], o_ref) < 1e-12
    assert rel_err(res["final_state"], fin_ref) < 1e-12


@pytest.mark.parametrize("M", [1, 2, 3, 4])
def test_bruteforce_transition_matrices(M):
    """Token loop == product of per-token affine maps built with matrix products (tiny inputs)."""
    w = make_custom([3, 8, 1], 2, 4, M, seed=20 + M, decay=0.5, init_sigma=0.7, normalised=False)
    for l2 in (False, True):
        res = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, 0.37,
                             use_qk_l2norm=l2, initial_state=w.initial_state)
        o_ref, fin_ref, _ = transition_bruteforce(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, 0.37,
                                                  S0_vmajor=w.initial_state, l2norm=l2)
        assert rel_err(res["o"], o_ref) < 1e-12
        assert rel_err(res["final_state"], fin_ref) < 1e-12


def _signed_four_hot(gen, rows, H, d):
    """Rows with exactly four entries of +-1/2 (exact unit norm in bf16)."""
    out = torch.zeros(rows, H, d)
    for r in range(rows):
        for h in range(H):
            idx = torch.randperm(d, generator=gen)[:4]
            sgn = torch.randint(0, 2, (4,), generator=gen).float() * 2 - 1
            out[r, h, idx] = 0.5 * sgn
    return out.to(torch.bfloat16)


@pytest.mark.parametrize("M", [1, 2, 3])
def test_householder_projection(M):
    """beta = 1 and unit k: after each token S k_last = v_last (projection property of the update).
    With q_t = k_{t,M-1} and scale 1 the readout returns v_{t,M-1} exactly."""
    gen = torch.Generator().manual_seed(5 + M)
    w = make_custom([9, 30], 3, 16, M, seed=40 + M, decay=0.4, init_sigma=0.3)
    k = _signed_four_hot(gen, w.T * M, 3, 16)
    q = k[M - 1::M].clone()
    beta = torch.ones(w.T * M, 3)
    res = oracle.forward(q, k, w.v, w.g, beta, w.cu_seqlens, M, 1.0, initial_state=w.initial_state)
    np.testing.assert_allclose(res["o"], f64(w.v)[M - 1::M], rtol=0, atol=1e-12)


@pytest.mark.parametrize("M", [1, 3])
def test_beta_zero_closed_form(M):
    """beta = 0 leaves only the decay: o_t = scale * (prod_{s<=t} alpha_s) S0 q_t."""
    w = make_custom([7, 40], 2, 8, M, seed=60 + M, decay=0.2, init_sigma=1.0)
    beta = torch.zeros(w.T * M, 2)
    res = oracle.forward(w.q, w.k, w.v, w.g, beta, w.cu_seqlens, M, w.scale, initial_state=w.initial_state)
    g, q, S0 = f64(w.g), f64(w.q), f64(w.initial_state)
    cu = w.cu_seqlens.tolist()
    for i in range(w.N):
        for h in range(2):
            logp = 0.0
            for t in range(cu[i], cu[i + 1]):
                logp += g[t, h]
                np.testing.assert_allclose(res["o"][t, h], w.scale * math.exp(logp) * (S0[i, h] @ q[t, h]),
                                           rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(res["final_state"][i, h], math.exp(logp) * S0[i, h], rtol=1e-12)


def test_copy_indexing():
    """M = 3 with beta = 0 on copies 1, 2 equals M = 1 on copy 0: the decay acts once per real
    token and the copies of token t sit at rows t*M .. t*M+M-1."""
    w = make_custom([13, 70], 2, 8, 3, seed=77, decay=0.3, init_sigma=0.5)
    beta = w.beta.clone()
    beta.view(w.T, 3, 2)[:, 1:, :] = 0
    res3 = oracle.forward(w.q, w.k, w.v, w.g, beta, w.cu_seqlens, 3, w.scale, initial_state=w.initial_state)
    res1 = oracle.forward(w.q, w.k[0::3].contiguous(), w.v[0::3].contiguous(), w.g, beta[0::3].contiguous(),
                          w.cu_seqlens, 1, w.scale, initial_state=w.initial_state)
    np.testing.assert_allclose(res3["o"], res1["o"], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(res3["final_state"], res1["final_state"], rtol=1e-13, atol=1e-15)
    # and the copies are not interchangeable: moving beta to copy 2 changes the result
    beta2 = w.beta.clone()
    beta2.view(w.T, 3, 2)[:, :2, :] = 0
    res_other = oracle.forward(w.q, w.k, w.v, w.g, beta2, w.cu_seqlens, 3, w.scale, initial_state=w.initial_state)
    assert rel_err(res_other["o"], res1["o"]) > 1e-3


def test_linearity_in_state_and_values():
    """For fixed k, beta, g the map (S0, V) -> o is linear."""
    w = make_custom([20, 33], 2, 8, 2, seed=90, decay=0.2, init_sigma=0.5)
    zero_v = torch.zeros_like(w.v)
    a = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, 2, w.scale, initial_state=w.initial_state)
    b = oracle.forward(w.q, w.k, zero_v, w.g, w.beta, w.cu_seqlens, 2, w.scale, initial_state=w.initial_state)
    c = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, 2, w.scale, initial_state=None)
    np.testing.assert_allclose(a["o"], b["o"] + c["o"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(a["final_state"], b["final_state"] + c["final_state"], rtol=1e-11, atol=1e-12)


def test_varlen_packing_equals_separate_runs():
    """Packed THD input: each sequence is independent of its neighbours."""
    w = make_custom([10, 0, 64, 129], 2, 8, 2, seed=101, decay=0.2, init_sigma=0.5)
    packed = _run(w)
    cu = w.cu_seqlens.tolist()
    for i, L in enumerate(w.lengths):
        t0, t1 = cu[i], cu[i + 1]
        sub = oracle.forward(w.q[t0:t1], w.k[2 * t0:2 * t1], w.v[2 * t0:2 * t1], w.g[t0:t1], w.beta[2 * t0:2 * t1],
                             [0, L], 2, w.scale, initial_state=w.initial_state[i:i + 1])
        np.testing.assert_array_equal(packed["o"][t0:t1], sub["o"])
        np.testing.assert_array_equal(packed["final_state"][i], sub["final_state"][0])
    # the empty sequence copies its initial state through
    np.testing.assert_array_equal(packed["final_state"][1], f64(w.initial_state[1]))


@pytest.mark.parametrize("split", [64, 100, 1])
def test_resume_and_chunk_states(split):
    """Splitting a sequence and feeding part A's final state to part B equals one run; the
    chunk-state row c equals the final state of the first 64 c tokens."""
    M, L = 2, 200
    w = make_custom([L], 2, 8, M, seed=120, decay=0.1, init_sigma=0.5, chunk_states=True)
    whole = _run(w)
    a = oracle.forward(w.q[:split], w.k[:M * split], w.v[:M * split], w.g[:split], w.beta[:M * split],
                       [0, split], M, w.scale, initial_state=w.initial_state)
    b = oracle.forward(w.q[split:], w.k[M * split:], w.v[M * split:], w.g[split:], w.beta[M * split:],
                       [0, L - split], M, w.scale, initial_state=torch.from_numpy(a["final_state"]).float())
    # part B starts from the fp32 rounding of part A's state, hence the tolerance
    assert rel_err(np.concatenate([a["o"], b["o"]]), whole["o"]) < 1e-6
    assert rel_err(b["final_state"], whole["final_state"]) < 1e-6
    cs = whole["chunk_states"]
    assert cs.shape[0] == (L + 63) // 64
    np.testing.assert_array_equal(cs[0], f64(w.initial_state[0]))
    for c in range(1, cs.shape[0]):
        pre = oracle.forward(w.q[:64 * c], w.k[:M * 64 * c], w.v[:M * 64 * c], w.g[:64 * c], w.beta[:M * 64 * c],
                             [0, 64 * c], M, w.scale, initial_state=w.initial_state)
        np.testing.assert_array_equal(cs[c], pre["final_state"][0])


def test_chunk_states_match_bruteforce_entering_states():
    """Chunk-state rows against the brute-force entering state of token 64 c (multi-sequence)."""
    M = 3
    w = make_custom([65, 3, 130], 1, 4, M, seed=130, decay=0.3, init_sigma=0.5, chunk_states=True)
    res = _run(w)
    _, _, enter = transition_bruteforce(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, w.scale,
                                        S0_vmajor=w.initial_state)
    co = res["chunk_offsets"]
    cu = w.cu_seqlens.tolist()
    for i, L in enumerate(w.lengths):
        for c in range((L + 63) // 64):
            assert rel_err(res["chunk_states"][co[i] + c], enter[cu[i] + 64 * c]) < 1e-12


def test_state_cache_slots():
    """State cache: slot >= 0 read and written in place, slot -1 is padding (zero start,
    nothing written), other slots untouched."""
    w = make_custom([30, 5, 70, 12], 2, 8, 2, seed=140, decay=0.2, cache_slots=9, padding_slots=1)
    res = _run(w)
    sidx = w.state_indices.tolist()
    cache = f64(w.state)
    used = {s for s in sidx if s >= 0}
    for s in range(9):
        if s not in used:
            np.testing.assert_array_equal(res["state_out"][s], cache[s])
    for i, s in enumerate(sidx):
        init = None if s < 0 else w.state[s:s + 1]
        t0, t1 = w.cu_seqlens[i].item(), w.cu_seqlens[i + 1].item()
        ref = oracle.forward(w.q[t0:t1], w.k[2 * t0:2 * t1], w.v[2 * t0:2 * t1], w.g[t0:t1], w.beta[2 * t0:2 * t1],
                             [0, t1 - t0], 2, w.scale, initial_state=init)
        np.testing.assert_array_equal(res["o"][t0:t1], ref["o"])
        if s >= 0:
            np.testing.assert_array_equal(res["state_out"][s], ref["final_state"][0])
    assert -1 in sidx


def _read_desc_cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "descriptors_varlen.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        if key == "case":
            cur = {"name": vals[0]}
            cases.append(cur)
        else:
            cur[key] = [int(x) for x in vals]
    return cases


@pytest.mark.parametrize("case", _read_desc_cases(), ids=lambda c: c["name"])
def test_descriptors_golden(case):
    """Hand-computed descriptors, incl. ceil(L M / 64) != M ceil(L / 64)."""
    L, M = case["lengths"], case["M"][0]
    cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
    ci, cid, co, cod = oracle.descriptors(cu, M)
    assert ci.shape[0] == case["nt_pad"][0] and cid.shape[0] == case["ntdp_pad"][0]
    np.testing.assert_array_equal(co, case["chunk_offsets"])
    np.testing.assert_array_equal(cod, case["chunk_offsets_dp"])
    np.testing.assert_array_equal(ci.ravel(), case["chunk_indices"])
    np.testing.assert_array_equal(cid.ravel(), case["chunk_indices_dp"])


def test_descriptor_counts_closed_form():
    """Counts are sums of ceilings; the shape-only padding bounds hold for any lengths."""
    rng = np.random.default_rng(7)
    for _ in range(50):
        n = int(rng.integers(1, 12))
        L = rng.integers(0, 700, n)
        M = int(rng.integers(1, 9))
        cu = np.concatenate([[0], np.cumsum(L)]).astype(np.int64)
        ci, cid, co, cod = oracle.descriptors(cu, M)
        assert co[-1] == sum(-(-x // 64) for x in L)
        assert cod[-1] == sum(-(-(x * M) // 64) for x in L)
        assert (ci[co[-1]:] == -1).all() and (cid[cod[-1]:] == -1).all()
        for i in range(n):
            rows = ci[co[i]:co[i + 1]]
            assert (rows[:, 0] == i).all() and (rows[:, 1] == np.arange(len(rows))).all()


def test_decay_cumsum():
    """Stage-1 cumsum: constant g gives G2 = g log2(e) (number of token-start rows so far in the
    64-row expanded chunk); the sum restarts at each chunk of the expanded sequence."""
    M, L, a = 3, 50, -0.25
    cu = [0, L, L + 30]
    g = torch.full((L + 30, 1), a)
    G2 = oracle.decay_cumsum(cu, g, 1, M)
    for i in range(2):
        r0, r1 = cu[i] * M, cu[i + 1] * M
        for r in range(r0, r1):
            p = (r - r0) % 64
            start = r - p
            n_tok_rows = sum(1 for s in range(start, r + 1) if s % M == 0)
            assert G2[r, 0] == pytest.approx(a * n_tok_rows / math.log(2), rel=1e-12)
    # exp2 of G2 at the last row of a chunk is the product of the token decays inside it
    w = make_custom([100], 1, 4, 2, seed=3, decay=0.5)
    G2 = oracle.decay_cumsum(w.cu_seqlens, w.g, 1, 2)
    g = f64(w.g)[:, 0]
    assert 2.0 ** G2[63, 0] == pytest.approx(math.exp(g[:32].sum()), rel=1e-12)
    assert 2.0 ** G2[127, 0] == pytest.approx(math.exp(g[32:64].sum()), rel=1e-12)


# ---- input variants (FlashInfer page, parameters q, k, v, g, beta, initial_state) ----

def test_f16_widening_exhaustive():
    """The oracle's binary16 widening equals numpy's float16 -> float64 for all 65536 bit patterns."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.widen_f16(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("M", [1, 3])
def test_f16_inputs_bruteforce(M):
    """float16 q / k / v, bf16 g, beta and initial state: the oracle equals the transition-matrix
    formulation run on the same values (widened by torch)."""
    w = make_custom([3, 9, 1], 2, 4, M, seed=90 + M, decay=0.5, init_sigma=0.7, normalised=False,
                    qkv_dtype=torch.float16, g_dtype=torch.bfloat16, beta_dtype=torch.float16,
                    state_dtype=torch.bfloat16)
    assert w.q.dtype == torch.float16 and w.initial_state.dtype == torch.bfloat16
    for l2 in (False, True):
        res = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, 0.41, use_qk_l2norm=l2,
                             initial_state=w.initial_state)
        o_ref, fin_ref, _ = transition_bruteforce(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, 0.41,
                                                  S0_vmajor=w.initial_state, l2norm=l2)
        assert rel_err(res["o"], o_ref) < 1e-12
        assert rel_err(res["final_state"], fin_ref) < 1e-12
    # a float16 pattern read as bf16 is a different number: the element type is honoured
    res_bf = oracle.forward(w.q.view(torch.bfloat16), w.k.view(torch.bfloat16), w.v.view(torch.bfloat16), w.g,
                            w.beta, w.cu_seqlens, M, 0.41, initial_state=w.initial_state)
    assert not np.allclose(res_bf["o"], o_ref)


@pytest.mark.parametrize("heads", [(2, 2, 4), (4, 2, 2), (4, 4, 2), (1, 1, 3)])
def test_grouped_heads_equal_repeated_heads(heads):
    """Head counts (Hq, Hk, Hv) below the state count H = max(Hq, Hv): the result equals the run on
    inputs whose heads are repeated explicitly, state head h taking head h // (H // Hx) of each."""
    hq, hk, hv = heads
    H = max(hq, hv)
    w = make_custom([5, 11], H, 4, 2, seed=130 + hq * 7 + hv, decay=0.4, init_sigma=0.5, normalised=False,
                    hq=hq, hk=hk, hv=hv)
    assert w.q.shape[1] == hq and w.k.shape[1] == hk and w.v.shape[1] == hv
    for l2 in (False, True):
        res = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, 2, 0.5, use_qk_l2norm=l2,
                             initial_state=w.initial_state)
        rep = [t.repeat_interleave(H // t.shape[1], dim=1) for t in (w.q, w.k, w.v)]
        o_ref, fin_ref, _ = transition_bruteforce(*rep, w.g, w.beta, w.cu_seqlens, 2, 0.5,
                                                  S0_vmajor=w.initial_state, l2norm=l2)
        assert rel_err(res["o"], o_ref) < 1e-12
        assert rel_err(res["final_state"], fin_ref) < 1e-12


@pytest.mark.parametrize("g_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_linear_alpha_gate(g_dtype):
    """g given as alpha in linear space multiplies the state by alpha itself: equal to the log-gate
    formulation at g = ln(alpha), and with beta = 0 to scale * (prod alpha) S0 q."""
    w = make_custom([6, 20], 2, 4, 2, seed=150, decay=0.6, init_sigma=0.8, normalised=False,
                    g_is_alpha=True, g_dtype=g_dtype)
    assert w.g_is_alpha and float(w.g.float().min()) > 0 and float(w.g.float().max()) <= 1
    res = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, 2, w.scale, initial_state=w.initial_state,
                         g_is_alpha=True)
    log_g = np.log(f64(w.g))
    o_ref, fin_ref, _ = transition_bruteforce(w.q, w.k, w.v, log_g, w.beta, w.cu_seqlens, 2, w.scale,
                                              S0_vmajor=w.initial_state)
    assert rel_err(res["o"], o_ref) < 1e-12
    assert rel_err(res["final_state"], fin_ref) < 1e-12
    beta0 = torch.zeros(w.T * 2, 2)
    res0 = oracle.forward(w.q, w.k, w.v, w.g, beta0, w.cu_seqlens, 2, w.scale, initial_state=w.initial_state,
                          g_is_alpha=True)
    a, q, S0 = f64(w.g), f64(w.q), f64(w.initial_state)
    cu = w.cu_seqlens.tolist()
    for i in range(w.N):
        for h in range(2):
            p = 1.0
            for t in range(cu[i], cu[i + 1]):
                p *= a[t, h]
                np.testing.assert_allclose(res0["o"][t, h], w.scale * p * (S0[i, h] @ q[t, h]), rtol=1e-12,
                                           atol=1e-14)


def test_transfer_pair_affine_in_state():
    """Over a sequence the state map is affine: S_end(S0) = S0 Phi + B, B the run from a zero
    state and Phi the run from the identity with v = 0 (the pair a sequence-sharded prefill
    exchanges; blog post "Attention Cache and Sequence Parallelism", passing state instead of
    KV).  Phi is checked against the product of the per-token transition matrices
    alpha_t prod_j (I - beta_j k_j k_j^T), built here directly; an empty sequence has B = 0,
    Phi = I."""
    M, H, d = 3, 2, 8
    w = make_custom([37, 0, 70], H, d, M, seed=140, decay=0.2, init_sigma=0.5)
    N = 3
    whole = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, w.scale, initial_state=w.initial_state)
    B = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, w.scale)["final_state"]
    eye = torch.eye(d).expand(N, H, d, d).contiguous()
    Phi = oracle.forward(w.q, w.k, torch.zeros_like(w.v), w.g, w.beta, w.cu_seqlens, M, w.scale,
                         initial_state=eye)["final_state"]
    S0 = f64(w.initial_state)
    np.testing.assert_allclose(whole["final_state"], S0 @ Phi + B, rtol=1e-10, atol=1e-12)
    np.testing.assert_array_equal(B[1], 0.0)
    np.testing.assert_array_equal(Phi[1], np.broadcast_to(np.eye(d), (H, d, d)))
    k, g, beta = f64(w.k), f64(w.g), f64(w.beta)
    cu = w.cu_seqlens.tolist()
    for i in (0, 2):
        for h in range(H):
            P = np.eye(d)
            for t in range(cu[i], cu[i + 1]):
                A = math.exp(g[t, h]) * np.eye(d)
                for j in range(M):
                    r = t * M + j
                    A = A @ (np.eye(d) - beta[r, h] * np.outer(k[r, h], k[r, h]))
                P = P @ A
            np.testing.assert_allclose(Phi[i, h], P, rtol=1e-10, atol=1e-13)


def test_transfer_pairs_chain_over_shards():
    """Cutting a sequence into consecutive shards at token boundaries: chaining the shards'
    pairs, S_{r+1} = S_r Phi_r + B_r from the initial state, gives every shard's entering state,
    and running each shard from it reproduces the whole run."""
    M, H, d, L = 2, 2, 8, 150
    w = make_custom([L], H, d, M, seed=141, decay=0.1, init_sigma=0.5)
    whole = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, M, w.scale, initial_state=w.initial_state)
    cuts = [0, 41, 41, 97, L]  # one empty shard
    S = f64(w.initial_state)
    outs = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sl = dict(q=w.q[a:b], k=w.k[M * a:M * b], v=w.v[M * a:M * b], g=w.g[a:b], beta=w.beta[M * a:M * b])
        run = oracle.forward(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], [0, b - a], M, w.scale,
                             initial_state=torch.from_numpy(S).float())
        outs.append(run["o"])
        Bs = oracle.forward(sl["q"], sl["k"], sl["v"], sl["g"], sl["beta"], [0, b - a], M, w.scale)["final_state"]
        eye = torch.eye(d).expand(1, H, d, d).contiguous()
        Ph = oracle.forward(sl["q"], sl["k"], torch.zeros_like(sl["v"]), sl["g"], sl["beta"], [0, b - a], M, w.scale,
                            initial_state=eye)["final_state"]
        S = S @ Ph + Bs
    # the shards start from fp32 roundings of the chained state, hence the tolerance
    assert rel_err(np.concatenate(outs), whole["o"]) < 1e-6
    assert rel_err(S, whole["final_state"]) < 1e-6
