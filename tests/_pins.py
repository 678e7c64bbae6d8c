"""Independent formulations used to pin the oracle (numpy, float64, tiny inputs).

None of these shares code with the oracle or with the CUDA path.

* ``gdn_kmajor``: the single-token gated delta rule as the blog post
  "Attention Cache and Sequence Parallelism" writes it in its GDN section
  (K-major state S in R^{K x V}: Sbar = lambda S, vhat = Sbar^T k,
  e = beta (v - vhat), S = Sbar + k e^T, r = q^T S), with lambda = exp(g).
  The FlashInfer page states that num_householder == 1 is exactly the gated
  delta rule, so the oracle at n = 1 must agree with it (after transposing the
  state and applying the readout scale).
* ``transition_bruteforce``: each token written as an affine map of the state,
  S -> S A_t + B_t with A_t = alpha_t prod_j (I - beta_j k_j k_j^T) and
  B_t = sum_j beta_j v_j k_j^T prod_{j' > j} (I - beta_j' k_j' k_j'^T),
  built with explicit matrix products.
"""
from __future__ import annotations

import numpy as np
import torch

EPS = 1e-6  # the L2-normalisation reading shared with the oracle's contract


def f64(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().double().numpy()
    return np.asarray(x, dtype=np.float64)


def _norm(x, on):
    if not on:
        return x
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + EPS)


def gdn_kmajor(q, k, v, g, beta, cu, scale, S0_vmajor=None, l2norm=False):
    """M = 1 only. Returns (o [T,H,V], final [N,H,V,K]) with the state handed back V-major."""
    q, k, v = _norm(f64(q), l2norm), _norm(f64(k), l2norm), f64(v)
    T, H, K = q.shape
    V = v.shape[2]
    g = np.zeros((T, H)) if g is None else f64(g)
    beta = np.ones((T, H)) if beta is None else f64(beta)
    cu = [int(x) for x in cu]
    N = len(cu) - 1
    o = np.zeros((T, H, V))
    fin = np.zeros((N, H, V, K))
    for i in range(N):
        for h in range(H):
            S = np.zeros((K, V)) if S0_vmajor is None else f64(S0_vmajor)[i, h].T.copy()
            for t in range(cu[i], cu[i + 1]):
                lam = np.exp(g[t, h])
                Sbar = lam * S
                vhat = Sbar.T @ k[t, h]
                e = beta[t, h] * (v[t, h] - vhat)
                S = Sbar + np.outer(k[t, h], e)
                o[t, h] = scale * (q[t, h] @ S)
            fin[i, h] = S.T
    return o, fin


def transition_bruteforce(q, k, v, g, beta, cu, M, scale, S0_vmajor=None, l2norm=False):
    """Any M. Returns (o [T,H,V], final [N,H,V,K], entering states per token [T,H,V,K])."""
    q, k, v = _norm(f64(q), l2norm), _norm(f64(k), l2norm), f64(v)
    T, H, K = q.shape
    V = v.shape[2]
    g = np.zeros((T, H)) if g is None else f64(g)
    beta = np.ones((T * M, H)) if beta is None else f64(beta)
    cu = [int(x) for x in cu]
    N = len(cu) - 1
    I = np.eye(K)
    o = np.zeros((T, H, V))
    fin = np.zeros((N, H, V, K))
    enter = np.zeros((T, H, V, K))
    for i in range(N):
        for h in range(H):
            S = np.zeros((V, K)) if S0_vmajor is None else f64(S0_vmajor)[i, h].copy()
            for t in range(cu[i], cu[i + 1]):
                enter[t, h] = S
                P = [I - beta[t * M + j, h] * np.outer(k[t * M + j, h], k[t * M + j, h]) for j in range(M)]
                A = np.exp(g[t, h]) * I
                for j in range(M):
                    A = A @ P[j]
                B = np.zeros((V, K))
                for j in range(M):
                    term = beta[t * M + j, h] * np.outer(v[t * M + j, h], k[t * M + j, h])
                    for jj in range(j + 1, M):
                        term = term @ P[jj]
                    B = B + term
                S = S @ A + B
                o[t, h] = scale * (S @ q[t, h])
            fin[i, h] = S
    return o, fin, enter


def rel_err(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.linalg.norm(b), 1e-300)
    return float(np.linalg.norm(a - b) / den)
