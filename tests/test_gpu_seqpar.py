"""GPU parity of the sequence-sharded prefill's device steps against the float64 oracle.

Ranks hold consecutive token shards of every sequence.  Each computes its shard's transfer
pairs (B: the state after the shard from zero; Phi: from the identity with v = 0), the pairs
are exchanged, each rank chains the pairs of the ranks before it onto the initial state and
runs its shard from there.  One GPU emulates the ranks one after another (plain launches in
order, no kernel waiting on another); the exchange itself is covered by the gloo tests.
"""
import numpy as np
import pytest
import torch

import chunked_gated_deltaproduct_gb300 as pkg
import oracle
from gdp_workloads import make_custom
from tests._parity import check_o, check_state

pytestmark = pytest.mark.gpu


def _shard(w, cuts, r, dev):
    M, cu = w.M, w.cu_seqlens.tolist()
    it, ie, lens = [], [], []
    for i in range(len(cu) - 1):
        a, b = cu[i] + cuts[i][r], cu[i] + cuts[i][r + 1]
        it += list(range(a, b))
        ie += list(range(M * a, M * b))
        lens.append(b - a)
    it, ie = torch.tensor(it, dtype=torch.long), torch.tensor(ie, dtype=torch.long)
    cu_l = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
    return dict(q=w.q[it].to(dev), k=w.k[ie].to(dev), v=w.v[ie].to(dev), g=w.g[it].to(dev),
                beta=w.beta[ie].to(dev), cu=cu_l.to(dev), lens=lens)


CASES = {
    # name: (workload kwargs, per-sequence shard boundaries for R ranks)
    "m2_d128_two_ranks": (dict(lengths=[1000, 300], H=4, d=128, M=2, init_sigma=0.1),
                          [[0, 421, 1000], [0, 0, 300]]),
    "m2_d128_three_ranks": (dict(lengths=[1000, 300], H=4, d=128, M=2, init_sigma=0.1),
                            [[0, 333, 334, 1000], [0, 150, 300, 300]]),
    "m3_d64_l2norm_four_ranks": (dict(lengths=[700, 129], H=2, d=64, M=3, normalised=False, use_qk_l2norm=True,
                                      init_sigma=0.2),
                                 [[0, 21, 22, 400, 700], [0, 64, 65, 129, 129]]),
    "f16_two_ranks": (dict(lengths=[900], H=2, d=128, M=2, init_sigma=0.2, qkv_dtype=torch.float16),
                      [[0, 512, 900]]),
}


def _run_sharded(w, cuts, dev):
    R = len(cuts[0]) - 1
    shards = [_shard(w, cuts, r, dev) for r in range(R)]
    pairs = torch.stack([pkg.chunk_gated_delta_product_transfer(s["q"], s["k"], s["v"], s["g"], s["beta"], s["cu"],
                                                                 w.M, w.scale, w.use_qk_l2norm) for s in shards])
    s0 = w.initial_state.to(dev).float().contiguous()
    chain = pkg.chain_states(s0, pairs[:, 1].contiguous(), pairs[:, 0].contiguous())  # [R + 1, N, H, V, K]
    o = torch.empty((w.T, w.H, w.d), dtype=w.q.dtype, device=dev)
    cu = w.cu_seqlens.tolist()
    fin = None
    for r, s in enumerate(shards):
        o_r, fin = pkg.chunk_gated_delta_product(s["q"], s["k"], s["v"], s["g"], s["beta"], s["cu"], w.M, w.scale,
                                                 initial_state=chain[r].contiguous(), output_final_state=True,
                                                 use_qk_l2norm_in_kernel=w.use_qk_l2norm)
        pos = 0
        for i, n in enumerate(s["lens"]):
            o[cu[i] + cuts[i][r]:cu[i] + cuts[i][r + 1]] = o_r[pos:pos + n]
            pos += n
    torch.cuda.synchronize()
    return pairs, chain, o, fin, shards


@pytest.mark.parametrize("name", sorted(CASES))
def test_sequence_sharded_prefill_emulated(cuda_device, name):
    kw, cuts = CASES[name]
    w = make_custom(seed=400 + sorted(CASES).index(name), **kw)
    pairs, chain, o, fin, _ = _run_sharded(w, cuts, cuda_device)
    ref = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale, use_qk_l2norm=w.use_qk_l2norm,
                         initial_state=w.initial_state)
    check_o(o.float().cpu(), ref["o"])
    check_state(fin.cpu(), ref["final_state"], label="final state (last shard)")
    check_state(chain[-1].cpu(), ref["final_state"], label="final state (chained pairs)")


def test_transfer_pairs_against_oracle(cuda_device):
    """B = the state after each sequence from zero, Phi = from the identity with v = 0; an empty
    sequence gives B = 0 and Phi = I exactly.  B is a state and meets the state tolerance.  Phi
    is not an output of the pages: it is the scan run with no fresh input, so nothing is
    forgotten -- every chunk's error stays in it.  The MMAs truncate their tf32 operands (10
    explicit mantissa bits: relative error below 2^-10, one-sided), so over n chunks the errors
    add up to at most about n 2^-10 per (sequence, head), rel L2 (measured: 6.2e-3 for 33 chunks
    against this 3.2e-2).  What the pairs feed -- the sharded prefill's outputs and states -- meets
    the pages' tolerances (test above)."""
    w = make_custom([700, 0, 230], 2, 128, 3, seed=420, decay=0.05)
    d = {k_: getattr(w, k_).to(cuda_device) for k_ in ("q", "k", "v", "g", "beta")}
    pairs = pkg.chunk_gated_delta_product_transfer(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                                   w.cu_seqlens.to(cuda_device), w.M, w.scale)
    torch.cuda.synchronize()
    B = oracle.forward(w.q, w.k, w.v, w.g, w.beta, w.cu_seqlens, w.M, w.scale)["final_state"]
    eye = torch.eye(w.d).expand(w.N, w.H, w.d, w.d).contiguous()
    Phi = oracle.forward(w.q, w.k, torch.zeros_like(w.v), w.g, w.beta, w.cu_seqlens, w.M, w.scale,
                         initial_state=eye)["final_state"]
    p = pairs.cpu()
    check_state(p[0][[0, 2]], B[[0, 2]], label="B")
    n = max((L * w.M + 63) // 64 for L in w.lengths)
    tol = n * 2.0 ** -10
    for i in (0, 2):
        for h in range(w.H):
            g_, r_ = p[1][i, h].double().numpy(), Phi[i, h]
            rel = np.linalg.norm(g_ - r_) / np.linalg.norm(r_)
            assert rel <= tol, (i, h, rel, tol)
    assert torch.count_nonzero(p[0][1]).item() == 0
    assert torch.equal(p[1][1], torch.eye(w.d).expand(w.H, w.d, w.d))


@pytest.mark.parametrize("d,steps", [(128, 5), (64, 3), (128, 0)])
def test_chain_states_against_float64(cuda_device, d, steps):
    """S_{j+1} = S_j Phi_j + B_j (fp32 FMA) against the same chain in float64."""
    gen = torch.Generator().manual_seed(430 + d + steps)
    N, H = 3, 2
    phi = torch.randn((steps, N, H, d, d), generator=gen) / d ** 0.5
    b = torch.randn((steps, N, H, d, d), generator=gen)
    s0 = torch.randn((N, H, d, d), generator=gen)
    out = pkg.chain_states(s0.to(cuda_device), phi.to(cuda_device), b.to(cuda_device)).cpu()
    ref = [s0.double()]
    for j in range(steps):
        ref.append(ref[-1] @ phi[j].double() + b[j].double())
    ref = torch.stack(ref)
    assert torch.equal(out[0], s0)
    err = (out.double() - ref).norm() / ref.norm()
    assert err < 2e-6, float(err)
    none = pkg.chain_states(None, phi.to(cuda_device), b.to(cuda_device)).cpu()  # S_0 = 0
    assert torch.count_nonzero(none[0]).item() == 0
    if steps:
        ref0 = [torch.zeros_like(s0, dtype=torch.float64)]
        for j in range(steps):
            ref0.append(ref0[-1] @ phi[j].double() + b[j].double())
        assert (none.double() - torch.stack(ref0)).norm() / torch.stack(ref0).norm() < 2e-6

