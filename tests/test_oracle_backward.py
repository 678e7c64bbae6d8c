"""Pins of the float64 backward oracle (``oracle.backward``).

The backward pass is the derivative of the forward recurrence (FlashInfer page
"flashinfer.gdp_prefill.chunk_gated_delta_product", display equation; blog post
"Attention Cache and Sequence Parallelism", section on passing state instead of
KV: training runs the recurrence in chunks and its backward dependence runs the
other way round).  The oracle takes that derivative step by step; here it is
checked against

* torch reverse-mode autograd through an independent float64 torch loop of the
  forward definition (every gradient, M = 1..4, with and without the in-kernel
  L2 norm, packed sequences, initial and final states);
* central finite differences of the C forward oracle itself in g, beta and the
  initial state (inputs on a 2^-20 grid, steps of 2^-12, so every perturbed
  input is exact in fp32);
* the closed form at beta = 0, where S_t = (prod alpha) S_0;
* linearity in the upstream gradients.

A set of planted mistakes in copies of the oracle's C source must each fail
one of these pins.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
import oracle.oracle as orc
from gdp_workloads import make_cotangents, make_custom

EPS = 1e-6


def _torch_forward(q, k, v, g, beta, cu, M, scale, l2norm, init):
    """The forward definition as a plain float64 torch loop (heads vectorised)."""
    T, H, K = q.shape
    V = v.shape[2]
    N = len(cu) - 1
    outs, fins = [], []

    def hat(x):
        return x / torch.sqrt((x * x).sum(-1, keepdim=True) + EPS) if l2norm else x

    for i in range(N):
        S = init[i].clone() if init is not None else torch.zeros(H, V, K, dtype=torch.float64)
        for t in range(int(cu[i]), int(cu[i + 1])):
            if g is not None:
                S = S * torch.exp(g[t])[:, None, None]
            for j in range(M):
                r = t * M + j
                kr = hat(k[r])
                b = beta[r] if beta is not None else torch.ones(H, dtype=torch.float64)
                vn = b[:, None] * (v[r] - torch.einsum("hvk,hk->hv", S, kr))
                S = S + vn[:, :, None] * kr[:, None, :]
            outs.append(scale * torch.einsum("hvk,hk->hv", S, hat(q[t])))
        fins.append(S)
    o = torch.stack(outs) if outs else torch.zeros(0, H, V, dtype=torch.float64)
    return o, torch.stack(fins)


def _autograd(w, d_out, d_fin):
    d = lambda x: None if x is None else x.detach().double().clone().requires_grad_(True)
    xs = {n: d(getattr(w, n)) for n in ("q", "k", "v", "g", "beta")}
    init = d(w.initial_state) if w.initial_state is not None else None
    o, fin = _torch_forward(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"], w.cu_seqlens.tolist(), w.M, w.scale,
                            w.use_qk_l2norm, init)
    loss = (o * d_out.double()).sum()
    if d_fin is not None:
        loss = loss + (fin * d_fin.double()).sum()
    named = [(n, x) for n, x in xs.items() if x is not None] + ([("initial_state", init)] if init is not None else [])
    grads = torch.autograd.grad(loss, [x for _, x in named])
    return {n: gr.numpy() for (n, _), gr in zip(named, grads)}, o.detach().numpy(), fin.detach().numpy()


def _oracle(w, d_out, d_fin, **kw):
    return oracle.backward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, d_out,
                           use_qk_l2norm=w.use_qk_l2norm, initial_state=w.initial_state, d_final_state=d_fin, **kw)


def _rel(a, b):
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


NAMES = {"q": "dq", "k": "dk", "v": "dv", "g": "dg", "beta": "dbeta", "initial_state": "d_initial_state"}


@pytest.mark.parametrize("M,l2norm", [(1, False), (2, True), (3, False), (4, True)])
def test_backward_matches_autograd(M, l2norm):
    w = make_custom([5, 9, 3, 0, 4], 2, 8, M, seed=10 + M, normalised=not l2norm, use_qk_l2norm=l2norm,
                    decay=0.3, init_sigma=0.3)
    d_out, d_fin = make_cotangents(w, seed=M)
    ref, o, fin = _autograd(w, d_out, d_fin)
    got = _oracle(w, d_out, d_fin)
    assert _rel(got["o"], o) < 1e-12 and _rel(got["final_state"], fin) < 1e-12
    for n, gr in ref.items():
        assert _rel(got[NAMES[n]], gr) < 1e-11, (n, _rel(got[NAMES[n]], gr))


def test_backward_across_checkpoint_blocks():
    """Sequences longer than the 64-token checkpoint blocks, no final-state gradient."""
    w = make_custom([70, 130], 1, 4, 2, seed=3, decay=0.05, init_sigma=0.2)
    d_out, _ = make_cotangents(w, seed=4, d_final_state=False)
    ref, _, _ = _autograd(w, d_out, None)
    got = _oracle(w, d_out, None)
    for n, gr in ref.items():
        assert _rel(got[NAMES[n]], gr) < 1e-10, (n, _rel(got[NAMES[n]], gr))


def _c_forward_loss(w, d_out, d_fin, g, beta, init):
    r = oracle.forward(w.q, w.k, w.v, g, beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                       initial_state=init)
    return float((r["o"] * d_out.double().numpy()).sum() + (r["final_state"] * d_fin.double().numpy()).sum())


@pytest.mark.parametrize("which", ["g", "beta", "initial_state"])
def test_backward_finite_differences_of_c_forward(which):
    w = make_custom([6, 11], 2, 8, 2, seed=21, use_qk_l2norm=True, normalised=False, decay=0.3, init_sigma=0.3)
    d_out, d_fin = make_cotangents(w, seed=22, quantum=2.0 ** -20)
    got = _oracle(w, d_out, d_fin)
    gen = torch.Generator().manual_seed(5)
    x = getattr(w, which)
    u = torch.randint(0, 2, x.shape, generator=gen).float() * 2 - 1
    h = 2.0 ** -12
    args = {"g": w.g, "beta": w.beta, "init": w.initial_state}
    key = "init" if which == "initial_state" else which
    plus, minus = dict(args), dict(args)
    plus[key] = (x.double() + h * u.double()).float()
    minus[key] = (x.double() - h * u.double()).float()
    assert torch.equal(plus[key].double() - minus[key].double(), 2 * h * u.double())  # exact steps
    fd = (_c_forward_loss(w, d_out, d_fin, **plus) - _c_forward_loss(w, d_out, d_fin, **minus)) / (2 * h)
    an = float((got[NAMES[which]] * u.double().numpy()).sum())
    assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (fd, an)


def test_backward_beta_zero_closed_form():
    """beta = 0: S_t = A_t S_0 with A_t = prod_{s<=t} alpha_s, o_t = scale A_t S_0 qhat_t, so
    dv = dk = 0, dq_t = scale A_t S_0^T do_t, dg_t = sum_{t'>=t} do_t'.o_t' + <dS_T, S_T> and
    dS_0 = sum_t scale A_t do_t qhat_t^T + A_T dS_T."""
    w = make_custom([9], 2, 4, 2, seed=31, decay=0.4, init_sigma=0.5)
    w.beta = torch.zeros_like(w.beta)
    d_out, d_fin = make_cotangents(w, seed=32)
    got = _oracle(w, d_out, d_fin)
    g = w.g.double().numpy()
    A = np.exp(np.cumsum(g, 0))  # [T, H]
    S0 = w.initial_state.double().numpy()[0]  # [H, V, K]
    q = w.q.double().numpy()
    do = d_out.double().numpy()
    dS = d_fin.double().numpy()[0]
    o = w.scale * A[:, :, None] * np.einsum("hvk,thk->thv", S0, q)
    ST = A[-1][:, None, None] * S0
    assert np.abs(got["dv"]).max() == 0 and np.abs(got["dk"]).max() == 0
    dq = w.scale * A[:, :, None] * np.einsum("hvk,thv->thk", S0, do)
    assert _rel(got["dq"], dq) < 1e-12
    rho = (do * o).sum(-1)  # [T, H]
    dg = np.cumsum(rho[::-1], 0)[::-1] + (dS * ST).sum((-1, -2))[None, :]
    assert _rel(got["dg"], dg) < 1e-12
    dS0 = w.scale * np.einsum("th,thv,thk->hvk", A, do, q) + A[-1][:, None, None] * dS
    assert _rel(got["d_initial_state"][0], dS0) < 1e-12


def test_backward_linear_in_upstream_gradients():
    w = make_custom([7, 4], 2, 8, 3, seed=41, init_sigma=0.2)
    d1, f1 = make_cotangents(w, seed=1)
    d2, f2 = make_cotangents(w, seed=2)
    a, b = _oracle(w, d1, f1), _oracle(w, d2, f2)
    c = _oracle(w, d1.double() + d2.double(), f1.double() + f2.double())
    for n in ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state"):
        assert _rel(c[n], a[n] + b[n]) < 1e-12, n


SRC = open(os.path.join(os.path.dirname(orc.__file__), "gdp_oracle.c")).read()
MUTANTS = {
    "decay_not_propagated": [("for (int64_t x = 0; x < KV; ++x) D[x] *= a;", "")],
    "dg_after_decay": [("if (dg) dg[t * H + h] = g ? acc : 0.0;\n                const double a = g ? exp(g[t * H + h]) : 1.0;\n"
                        "                for (int64_t x = 0; x < KV; ++x) D[x] *= a;",
                        "const double a = g ? exp(g[t * H + h]) : 1.0;\n                for (int64_t x = 0; x < KV; ++x) D[x] *= a;\n"
                        "                if (dg) dg[t * H + h] = g ? acc * a : 0.0;")],
    "dk_second_term_sign": [("acc += b * D[(int64_t)vv * K + d] * e[vv] - P[(int64_t)vv * K + d] * dvv[vv];",
                             "acc += b * D[(int64_t)vv * K + d] * e[vv] + P[(int64_t)vv * K + d] * dvv[vv];")],
    "dbeta_uses_v": [("db += e[vv] * acc;", "db += v[(r * H + h) * (int64_t)V + vv] * acc;")],
    "l2_projection_dropped": [("dk[(r * H + h) * (int64_t)K + d] = use_qk_l2norm ? dkh[d] / n - kr[d] * dot / (n * n * n) : dkh[d];",
                               "dk[(r * H + h) * (int64_t)K + d] = use_qk_l2norm ? dkh[d] / n : dkh[d];")],
    "readout_uses_state_before_update": [("acc += (P[(int64_t)vv * K + d] + b * e[vv] * kh[d]) * dOt[vv];",
                                          "acc += P[(int64_t)vv * K + d] * dOt[vv];")],
    "rows_of_token_forward_order": [("for (int j = M - 1; j >= 0; --j) {", "for (int j = 0; j < M; ++j) {")],
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_backward_mutant_is_caught(mutant, tmp_path):
    src = SRC
    for old, new in MUTANTS[mutant]:
        assert src.count(old) == 1, f"mutation anchor missing or ambiguous: {old!r}"
        src = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    real = orc._load()
    lib = ctypes.CDLL(str(so))
    for fname in ("gdp_oracle_forward", "gdp_oracle_descriptors", "gdp_oracle_decay_cumsum", "gdp_oracle_widen_f16",
                  "gdp_oracle_backward"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    pins = [lambda: test_backward_matches_autograd(2, True), lambda: test_backward_matches_autograd(3, False),
            test_backward_across_checkpoint_blocks, test_backward_beta_zero_closed_form]
    saved = orc._lib
    orc._lib = lib
    caught = False
    try:
        for fn in pins:
            try:
                fn()
            except (AssertionError, ValueError):
                caught = True
                break
    finally:
        orc._lib = saved
    assert caught, f"no pin caught the planted mistake {mutant}"
