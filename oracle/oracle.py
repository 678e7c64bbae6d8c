"""ctypes loader for the float64 C oracle (``gdp_oracle.c``).

TEST INFRASTRUCTURE ONLY (tests, smoke check, CPU baseline of the bench).  The
shared object is compiled from ``gdp_oracle.c`` with the system C compiler on
first use (or by ``__graft_entry__.build()``) into ``oracle/_build/``.

Method sources, cited by page and section:
  * FlashInfer API page "flashinfer.gdp_prefill.chunk_gated_delta_product",
    display equation and parameters k, v, beta, initial_state, cu_seqlens,
    use_qk_l2norm_in_kernel, scale: the per-token recurrence and tensor contract.
  * Megatron-Core API page "core.ssm.ops.gdp.chunk", stage list and parameters
    g, chunk_indices, chunk_indices_dp, chunk_offsets, state, state_indices,
    return_chunk_states: log decays, the two 64-row chunkings, descriptors,
    chunk-state rows and the in-place state cache.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

CHUNK = 64
L2_EPS = 1e-6

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdp_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libgdp_oracle.so")
_lock = threading.Lock()
_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math) if stale."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if stale:
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build_oracle())
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            lib.gdp_oracle_forward.restype = ctypes.c_int
            lib.gdp_oracle_forward.argtypes = [
                i64, i64, i32, i32, i32, i32,  # T N H K V M
                i32, i32, i32, i32, i32,  # Hq Hk Hv qkv_f16 g_is_alpha
                P,  # cu_seqlens
                P, P, P,  # q k v
                P, P, dbl, i32,  # g beta scale l2norm
                P,  # initial_state
                P, P, i64,  # state_in state_indices num_slots
                P,  # chunk_offsets
                P,  # head_mask
                P, P, P, P,  # o final state_out chunk_states
                i32,
            ]
            lib.gdp_oracle_descriptors.restype = ctypes.c_int
            lib.gdp_oracle_descriptors.argtypes = [P, i64, i32, P, i64, P, i64, P, P]
            lib.gdp_oracle_widen_f16.restype = ctypes.c_double
            lib.gdp_oracle_widen_f16.argtypes = [ctypes.c_uint16]
            lib.gdp_oracle_decay_cumsum.restype = ctypes.c_int
            lib.gdp_oracle_decay_cumsum.argtypes = [i64, i64, i32, i32, P, P, P]
            lib.gdp_oracle_backward.restype = ctypes.c_int
            lib.gdp_oracle_backward.argtypes = [
                i64, i64, i32, i32, i32, i32,  # T N H K V M
                P,  # cu_seqlens
                P, P, P, P, P, dbl, i32,  # q k v g beta scale l2norm
                P, P, P,  # initial_state d_output d_final_state
                P, P, P, P, P, P,  # dq dk dv dg dbeta d_initial_state
                P, P,  # o final_state
                i32,
            ]
            _lib = lib
    return _lib


def oracle_threads() -> int:
    """Threads the oracle uses: the CPU cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _half_bits(x):
    """bf16 / float16 tensor (torch), or a uint16 array of bf16 bit patterns ->
    (contiguous uint16 bit patterns, 1 if float16 else 0)."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.float16:
            return np.ascontiguousarray(x).view(np.uint16), 1
        assert x.dtype == np.uint16
        return np.ascontiguousarray(x), 0
    import torch

    assert x.dtype in (torch.bfloat16, torch.float16), x.dtype
    bits = np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))
    return bits, int(x.dtype == torch.float16)


def _bf16_bits(x) -> np.ndarray:
    """bf16 tensor (torch) or uint16 array -> contiguous uint16 bit patterns."""
    bits, f16 = _half_bits(x)
    assert not f16
    return bits


def _f32(x):
    """fp32 copy of a float32 / bfloat16 / float16 input (every such value is an
    fp32 value, so the widening is exact)."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        assert x.dtype in (np.float32, np.float16, np.float64), x.dtype
        return np.ascontiguousarray(x, dtype=np.float32)
    return np.ascontiguousarray(x.detach().cpu().float().numpy())


def widen_f16(bits: int) -> float:
    """The oracle's binary16 -> float64 widening of one bit pattern (for its pin)."""
    return float(_load().gdp_oracle_widen_f16(int(bits)))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def descriptors(cu_seqlens, M: int, nt_pad: int | None = None, ntdp_pad: int | None = None):
    """Descriptors on the host: (chunk_indices [nt_pad,2], chunk_indices_dp [ntdp_pad,2],
    chunk_offsets [N+1], chunk_offsets_dp [N+1]), int32.  Default padding is the
    shape-only bound floor((T + 63 N) / 64) (resp. M*T)."""
    lib = _load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    T = int(cu[-1]) if N > 0 else 0
    if nt_pad is None:
        nt_pad = (T + (CHUNK - 1) * N) // CHUNK
    if ntdp_pad is None:
        ntdp_pad = (M * T + (CHUNK - 1) * N) // CHUNK
    ci = np.empty((max(nt_pad, 0), 2), np.int32)
    cid = np.empty((max(ntdp_pad, 0), 2), np.int32)
    co = np.empty(N + 1, np.int32)
    cod = np.empty(N + 1, np.int32)
    rc = lib.gdp_oracle_descriptors(_ptr(cu), N, M, _ptr(ci), nt_pad, _ptr(cid), ntdp_pad, _ptr(co), _ptr(cod))
    if rc != 0:
        raise ValueError(f"gdp_oracle_descriptors failed ({rc})")
    return ci, cid, co, cod


def decay_cumsum(cu_seqlens, g, H: int, M: int) -> np.ndarray:
    """Base-2 within-chunk cumulative decay of the expanded stream, [T*M, H] float64."""
    lib = _load()
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    T = int(cu[-1]) if N > 0 else 0
    g32 = _f32(g)
    out = np.zeros((T * M, H), np.float64)
    lib.gdp_oracle_decay_cumsum(T, N, H, M, _ptr(cu), _ptr(g32), _ptr(out))
    return out


def forward(q, k, v, g, beta, cu_seqlens, num_householder: int, scale: float,
            use_qk_l2norm: bool = False, initial_state=None, state=None, state_indices=None,
            chunk_states: bool = False, heads=None, threads: int | None = None,
            want_o: bool = True, want_final: bool = True, g_is_alpha: bool = False):
    """Run the oracle.  q [T,Hq,K], k [T*M,Hk,K], v [T*M,Hv,V] bf16 or float16
    (all three the same type); g [T,H] (natural-log decay, or alpha itself when
    ``g_is_alpha``) and beta [T*M,H] fp32 / bf16 / float16 (or None); states
    V-major fp32 (an initial state may also be bf16).  H = max(Hq, Hv) and state
    head h reads q head h // (H // Hq), k head h // (H // Hk), v head
    h // (H // Hv).  ``heads``: iterable of state-head indices to compute
    (default all).  Returns a dict of float64 arrays: o [T,H,V], final_state
    [N,H,V,K], state_out [S,H,V,K] (cache mode: the pristine cache with every
    slot >= 0 replaced), chunk_states [NT,H,V,K] and chunk_offsets [N+1]."""
    lib = _load()
    M = int(num_householder)
    (qb, fq), (kb, fk), (vb, fv) = _half_bits(q), _half_bits(k), _half_bits(v)
    assert fq == fk == fv, "q, k and v must share one element type"
    T, Hq, K = qb.shape
    Hk, Hv, V = kb.shape[1], vb.shape[1], vb.shape[2]
    H = max(Hq, Hv)
    assert H % Hq == 0 and H % Hk == 0 and H % Hv == 0, (Hq, Hk, Hv)
    assert kb.shape == (T * M, Hk, K) and vb.shape == (T * M, Hv, V)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    g32, b32 = _f32(g), _f32(beta)
    init = _f32(initial_state)
    cache = _f32(state)
    assert g32 is None or g32.shape == (T, H), "g must be [T, H] with H = max(Hq, Hv)"
    assert b32 is None or b32.shape == (T * M, H), "beta must be [T*M, H]"
    assert init is None or init.shape == (N, H, V, K)
    assert cache is None or cache.shape[1:] == (H, V, K)
    sidx = None if state_indices is None else np.ascontiguousarray(np.asarray(state_indices, dtype=np.int32))
    num_slots = 0 if cache is None else cache.shape[0]
    co = None
    if chunk_states:
        co = np.empty(N + 1, np.int32)
        if lib.gdp_oracle_descriptors(_ptr(cu), N, M, None, 0, None, 0, _ptr(co), None) != 0:
            raise ValueError("cu_seqlens must be non-decreasing from 0")
    mask = None
    if heads is not None:
        mask = np.zeros(H, np.uint8)
        mask[list(heads)] = 1
    o = np.zeros((T, H, V), np.float64) if want_o else None
    fin = np.zeros((N, H, V, K), np.float64) if want_final else None
    st_out = cache.astype(np.float64) if cache is not None else None
    cs = np.zeros((int(co[-1]), H, V, K), np.float64) if chunk_states else None
    rc = lib.gdp_oracle_forward(
        T, N, H, K, V, M, Hq, Hk, Hv, fq, int(bool(g_is_alpha)),
        _ptr(cu), _ptr(qb), _ptr(kb), _ptr(vb), _ptr(g32), _ptr(b32),
        float(scale), int(bool(use_qk_l2norm)), _ptr(init), _ptr(cache), _ptr(sidx), num_slots,
        _ptr(co), _ptr(mask), _ptr(o), _ptr(fin), _ptr(st_out), _ptr(cs),
        int(threads if threads is not None else oracle_threads()))
    if rc != 0:
        raise ValueError(f"gdp_oracle_forward rejected its arguments ({rc})")
    return {"o": o, "final_state": fin, "state_out": st_out, "chunk_states": cs, "chunk_offsets": co}


def _f64(x):
    """float64 copy of a bf16 / float16 / fp32 / float64 tensor or array (exact widening), or None."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return np.ascontiguousarray(x, dtype=np.float64)
    return np.ascontiguousarray(x.detach().cpu().double().numpy())


def backward(q, k, v, g, beta, cu_seqlens, num_householder: int, scale: float, d_output,
             use_qk_l2norm: bool = False, initial_state=None, d_final_state=None,
             threads: int | None = None):
    """Reverse mode of the recurrence (``gdp_oracle_backward``): the gradients of a loss L
    with dL/do = d_output [T,H,V] and dL/dS_final = d_final_state [N,H,V,K] (None: 0) with
    respect to q [T,H,K], k [T*M,H,K], v [T*M,H,V], g [T,H] (natural-log decay), beta
    [T*M,H] and the initial state [N,H,V,K].  Heads are one-to-one.  Returns a dict of
    float64 arrays: dq, dk, dv, dg, dbeta, d_initial_state, plus the forward values o and
    final_state."""
    lib = _load()
    M = int(num_householder)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    T, H, K = qd.shape
    V = vd.shape[2]
    assert kd.shape == (T * M, H, K) and vd.shape == (T * M, H, V)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int64))
    N = cu.shape[0] - 1
    gd, bd, init, dout, dfin = _f64(g), _f64(beta), _f64(initial_state), _f64(d_output), _f64(d_final_state)
    assert dout.shape == (T, H, V)
    assert gd is None or gd.shape == (T, H)
    assert bd is None or bd.shape == (T * M, H)
    assert init is None or init.shape == (N, H, V, K)
    assert dfin is None or dfin.shape == (N, H, V, K)
    out = {
        "dq": np.zeros((T, H, K)), "dk": np.zeros((T * M, H, K)), "dv": np.zeros((T * M, H, V)),
        "dg": np.zeros((T, H)), "dbeta": np.zeros((T * M, H)), "d_initial_state": np.zeros((N, H, V, K)),
        "o": np.zeros((T, H, V)), "final_state": np.zeros((N, H, V, K)),
    }
    rc = lib.gdp_oracle_backward(
        T, N, H, K, V, M, _ptr(cu), _ptr(qd), _ptr(kd), _ptr(vd), _ptr(gd), _ptr(bd), float(scale),
        int(bool(use_qk_l2norm)), _ptr(init), _ptr(dout), _ptr(dfin),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dg"]), _ptr(out["dbeta"]),
        _ptr(out["d_initial_state"]), _ptr(out["o"]), _ptr(out["final_state"]),
        int(threads if threads is not None else oracle_threads()))
    if rc != 0:
        raise ValueError(f"gdp_oracle_backward rejected its arguments ({rc})")
    return out
