"""The chunk-form algebra the GPU kernels evaluate, checked on the CPU against the oracle.

The forward kernels (WY, scan) and the backward kernels (reverse scan, per-chunk gradients)
evaluate the recurrence of the FlashInfer API page "flashinfer.gdp_prefill.chunk_gated_delta_product"
(display equation) in 64-row chunks of the expanded stream, with formulas derived from the row
recurrence by algebra (the headers of gdp_wy_body.cuh, gdp_scan_body.cuh, gdp_backward.cu and
gdp_bwd_chunk_tc.cu state them).  Here the same formulas are written out in float64 numpy, one
chunk at a time, and compared with the float64 oracle, which steps the recurrence row by row and
takes the derivative step by step: a wrong sign, index or mask in a formula fails these tests at
~1e-9 relative, independently of any GPU.  Nothing here imports the CUDA path.
"""
import numpy as np
import pytest

import oracle
from gdp_workloads import make_cotangents, make_custom

CH = 64


def _rows(x):
    return x.detach().double().numpy()


def chunk_form(q, k, v, g, beta, M, scale, S0, dO, dS_fin, l2norm, mutate=None):
    """One sequence, one head.  q [L,K], k [L*M,K], v [L*M,V], g [L] (natural-log decay) or None,
    beta [L*M] or None, S0 [V,K], dO [L,V], dS_fin [V,K].  Returns the forward outputs and the
    gradients, all from the chunk formulas.  ``mutate`` plants one mistake (for the test that
    checks that the comparison catches it)."""
    L, K = q.shape
    R, V = L * M, v.shape[1]
    eps = oracle.L2_EPS
    nk = 1.0 / np.sqrt((k * k).sum(1) + eps) if l2norm else np.ones(R)
    nq = 1.0 / np.sqrt((q * q).sum(1) + eps) if l2norm else np.ones(L)
    kh, qh = k * nk[:, None], q * nq[:, None]
    gate = np.zeros(R)
    if g is not None:
        gate[0::M] = g
    b = np.ones(R) if beta is None else beta
    o = np.zeros((L, V))
    chunks = []
    S = S0.copy()
    for r0 in range(0, R, CH):
        r1 = min(R, r0 + CH)
        n = r1 - r0
        G = np.cumsum(gate[r0:r1])
        gam = np.exp(G)
        gC = gam[-1]
        Kc, Vc, bc = kh[r0:r1], v[r0:r1], b[r0:r1]
        ratio = gam[:, None] / gam[None, :]  # gamma_r / gamma_j
        Lm = np.tril(ratio * (Kc @ Kc.T), -1)
        T = np.linalg.inv(np.eye(n) + bc[:, None] * Lm)
        rhs = Vc - gam[:, None] * (Kc @ S.T)
        vt = T @ (bc[:, None] * rhs)
        e = rhs - Lm @ vt
        pl = np.array([p for p in range(n) if (r0 + p) % M == M - 1], dtype=np.int64)  # readout rows
        tok = (r0 + pl) // M
        Qp = qh[tok]
        mask = (np.arange(n)[None, :] <= pl[:, None]).astype(float)
        P = scale * mask * (gam[pl][:, None] / gam[None, :]) * (Qp @ Kc.T)
        o[tok] = scale * gam[pl][:, None] * (Qp @ S.T) + P @ vt
        chunks.append(dict(r0=r0, r1=r1, S=S.copy(), gam=gam, gC=gC, Kc=Kc, Vc=Vc, bc=bc, Lm=Lm, T=T, e=e,
                           vt=vt, pl=pl, tok=tok, Qp=Qp, P=P))
        S = gC * S + ((gC / gam)[:, None] * vt).T @ Kc
    S_fin = S
    # ---- backward: D = dL/dS at each chunk's exit, last chunk first ----
    dkh, dqh = np.zeros((R, K)), np.zeros((L, K))
    dv, dbeta = np.zeros((R, V)), np.zeros(R)
    D = dS_fin.copy()
    for c in reversed(chunks):
        gam, gC, Kc, bc, T, e, vt, pl, tok, Qp, P, Sc = (c[x] for x in
                                                       ("gam", "gC", "Kc", "bc", "T", "e", "vt", "pl", "tok", "Qp", "P", "S"))
        n = Kc.shape[0]
        dOp = dO[tok]
        Ktil = (gC / gam)[:, None] * Kc
        Zt = Ktil @ D.T + P.T @ dOp
        Delta = T.T @ Zt
        dvc = bc[:, None] * Delta
        idx = np.arange(n)
        gp = gam[pl]
        M1 = scale * (idx[:, None] <= pl[None, :]) * (gp[None, :] / gam[:, None]) * (e @ dOp.T)
        upper = (idx[None, :] >= idx[:, None]) if mutate == "m2_diagonal" else (idx[None, :] > idx[:, None])
        M2 = upper * (gam[None, :] / gam[:, None]) * (e @ dvc.T)
        M3 = (idx[None, :] < idx[:, None]) * (gam[:, None] / gam[None, :]) * (dvc @ vt.T)
        if mutate == "m3_sign":
            M3 = -M3
        M4 = (idx[None, :] <= pl[:, None]) * (gp[:, None] / gam[None, :]) * (dOp @ vt.T)
        dkh[c["r0"]:c["r1"]] = (bc[:, None] * ((gC / gam)[:, None] * (e @ D) + M1 @ Qp - M2 @ Kc)
                               - gam[:, None] * (dvc @ Sc) - M3 @ Kc)
        dqh[tok] += scale * (gp[:, None] * (dOp @ Sc) + M4 @ Kc)
        dv[c["r0"]:c["r1"]] = dvc
        dbeta[c["r0"]:c["r1"]] = (e * Delta).sum(1)
        W = T @ ((bc * gam)[:, None] * Kc)
        Qh = scale * gp[:, None] * Qp
        if mutate == "drop_readout_map":
            D = D @ (gC * np.eye(K) - Ktil.T @ W)
        elif mutate == "transposed_transition":
            D = (gC * np.eye(K) - Ktil.T @ W).T @ D.T + dOp.T @ (Qh - P @ W)
        else:
            D = D @ (gC * np.eye(K) - Ktil.T @ W) + dOp.T @ (Qh - P @ W)
    # the decay gradient needs no state: dg_t = <dS_T, S_T> + sum_{t' >= t} (dO_t' . o_t' - sum_j dv . v)
    term = (dO * o).sum(1) - (dv * v).sum(1).reshape(L, M).sum(1)
    dg = (dS_fin * S_fin).sum() + np.cumsum(term[::-1])[::-1]
    if l2norm:
        dk = nk[:, None] * (dkh - (kh * dkh).sum(1)[:, None] * kh)
        dq = nq[:, None] * (dqh - (qh * dqh).sum(1)[:, None] * qh)
    else:
        dk, dq = dkh, dqh
    return dict(o=o, final_state=S_fin, dq=dq, dk=dk, dv=dv, dbeta=dbeta, dg=dg, d_initial_state=D)


def _compare(w, d_out, d_fin):
    ref = oracle.backward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, d_out,
                          use_qk_l2norm=w.use_qk_l2norm, initial_state=w.initial_state, d_final_state=d_fin)
    cu = w.cu_seqlens.tolist()
    M = w.M
    for h in range(w.H):
        for i in range(w.N):
            t0, t1 = cu[i], cu[i + 1]
            if t1 == t0:
                continue
            S0 = np.zeros((w.d, w.d)) if w.initial_state is None else _rows(w.initial_state[i, h])
            dSf = np.zeros((w.d, w.d)) if d_fin is None else _rows(d_fin[i, h])
            got = chunk_form(_rows(w.q[t0:t1, h]), _rows(w.k[t0 * M:t1 * M, h]), _rows(w.v[t0 * M:t1 * M, h]),
                             None if w.g is None else _rows(w.g[t0:t1, h]),
                             None if w.beta is None else _rows(w.beta[t0 * M:t1 * M, h]),
                             M, w.scale, S0, _rows(d_out[t0:t1, h]), dSf, w.use_qk_l2norm)
            want = dict(o=ref["o"][t0:t1, h], final_state=ref["final_state"][i, h], dq=ref["dq"][t0:t1, h],
                        dk=ref["dk"][t0 * M:t1 * M, h], dv=ref["dv"][t0 * M:t1 * M, h],
                        dbeta=ref["dbeta"][t0 * M:t1 * M, h], dg=ref["dg"][t0:t1, h],
                        d_initial_state=ref["d_initial_state"][i, h])
            for name, x in want.items():
                if name == "dg" and w.g is None:
                    continue
                err = np.linalg.norm(got[name] - x) / max(np.linalg.norm(x), 1e-300)
                assert err < 1e-9, f"{name} (sequence {i}, head {h}): relative error {err:.3e}"


CASES = {
    # tokens per sequence, heads, head size, updates per token, keyword arguments
    "m2_several_chunks": ([100, 45], 2, 16, 2, dict(init_sigma=0.1)),
    "m3_chunks_split_tokens": ([70, 30], 1, 16, 3, dict(init_sigma=0.1, decay=0.3)),
    "m1_l2norm": ([150], 1, 8, 1, dict(normalised=False, use_qk_l2norm=True)),
    "m4_no_decay_no_beta": ([40, 17], 1, 8, 4, dict(with_g=False, with_beta=False, init_sigma=0.05)),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_chunk_form_matches_oracle(case):
    lengths, H, d, M, kw = CASES[case]
    w = make_custom(lengths, H, d, M, seed=300 + sorted(CASES).index(case), **kw)
    d_out, d_fin = make_cotangents(w, seed=301, dfin_sigma=0.5)
    _compare(w, d_out, d_fin)


def test_chunk_form_without_final_state_gradient():
    w = make_custom([90], 1, 8, 2, seed=310, init_sigma=0.1)
    d_out, _ = make_cotangents(w, seed=311, d_final_state=False)
    _compare(w, d_out, None)


@pytest.mark.parametrize("mutate", ["drop_readout_map", "transposed_transition", "m2_diagonal", "m3_sign"])
def test_chunk_form_detects_planted_mistakes(mutate):
    """The comparison has teeth: each planted mistake in the formulas (a dropped term, a
    transposed operand, a wrong mask, a wrong sign) disagrees with the oracle."""
    w = make_custom([130], 1, 8, 2, seed=320, init_sigma=0.1)
    d_out, d_fin = make_cotangents(w, seed=321, dfin_sigma=0.5)
    ref = oracle.backward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, d_out,
                          initial_state=w.initial_state, d_final_state=d_fin)
    args = (_rows(w.q[:, 0]), _rows(w.k[:, 0]), _rows(w.v[:, 0]), _rows(w.g[:, 0]), _rows(w.beta[:, 0]), w.M,
            w.scale, _rows(w.initial_state[0, 0]), _rows(d_out[:, 0]), _rows(d_fin[0, 0]), False)
    good, bad = chunk_form(*args), chunk_form(*args, mutate=mutate)
    names = ("dq", "dk", "dv", "dbeta", "d_initial_state")
    wants = {"dq": ref["dq"][:, 0], "dk": ref["dk"][:, 0], "dv": ref["dv"][:, 0], "dbeta": ref["dbeta"][:, 0],
             "d_initial_state": ref["d_initial_state"][0, 0]}
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert max(rel(good[n], wants[n]) for n in names) < 1e-9
    assert max(rel(bad[n], wants[n]) for n in names) > 1e-3
