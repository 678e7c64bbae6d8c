"""Thin ctypes binding of ``libgdp_gb300.so`` (argument marshalling only).

The names mirror the C ABI in ``include/gdp_prefill.h``: ``gdp_prefill_varlen``,
``gdp_prefill_varlen_profiled``, ``gdp_prefill_workspace_bytes``,
``gdp_prefill_varlen_backward``, ``gdp_backward_workspace_bytes``,
``gdp_build_descriptors``, ``gdp_last_error``, ``gdp_nt_pad``, ``gdp_ntdp_pad``.
``chunk_gated_delta_product`` wraps them with the keyword signature of the
pages (FlashInfer API page "flashinfer.gdp_prefill.chunk_gated_delta_product";
Megatron-Core API page "core.ssm.ops.gdp.chunk", function
chunk_gated_delta_product_varlen): torch supplies device memory and the
current stream, every step of the computation runs in the library's CUDA
kernels.  There is no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgdp_gb300.so")
DEBUG_LIB_PATH = os.path.join(_PKG, "libgdp_gb300_debug.so")  # the debug-bounds build

GDP_OK, GDP_ERR_INVALID_ARG, GDP_ERR_UNSUPPORTED, GDP_ERR_ALIAS, GDP_ERR_WORKSPACE, GDP_ERR_CUDA = range(6)
GDP_DEV_ERR_CU_SEQLENS, GDP_DEV_ERR_SLOT, GDP_DEV_ERR_DESC, GDP_DEV_ERR_TIMEOUT = 0x1, 0x2, 0x4, 0x8
GDP_DEV_ERR_BOUNDS = 0x10
BOUNDS_SITES = {1: "desc", 2: "wy_tile", 3: "wy_scalars", 4: "scan_order", 5: "scan_tile", 6: "scan_state",
                7: "scan_out", 8: "decode"}
GDP_DTYPE_DEFAULT, GDP_DTYPE_F32, GDP_DTYPE_BF16, GDP_DTYPE_F16 = range(4)
GDP_ABI_VERSION = 2
_DTYPE_CODE = {torch.float32: GDP_DTYPE_F32, torch.bfloat16: GDP_DTYPE_BF16, torch.float16: GDP_DTYPE_F16}
STATUS_NAMES = {0: "GDP_OK", 1: "GDP_ERR_INVALID_ARG", 2: "GDP_ERR_UNSUPPORTED", 3: "GDP_ERR_ALIAS",
                4: "GDP_ERR_WORKSPACE", 5: "GDP_ERR_CUDA"}

_vp, _i64, _int, _f32, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class GdpPrefillArgs(ctypes.Structure):
    """Mirror of ``gdp_prefill_args`` (field order and types of the header)."""
    _fields_ = [
        ("q", _vp), ("q_stride_t", _i64), ("q_stride_h", _i64),
        ("k", _vp), ("k_stride_t", _i64), ("k_stride_h", _i64),
        ("v", _vp), ("v_stride_t", _i64), ("v_stride_h", _i64),
        ("g", _vp), ("beta", _vp),
        ("cu_seqlens", _vp), ("cu_seqlens_int64", _int),
        ("T", _i64), ("N", _i64),
        ("H", _int), ("K", _int), ("V", _int), ("num_householder", _int),
        ("scale", _f32), ("use_qk_l2norm", _int),
        ("initial_state", _vp), ("state", _vp), ("state_indices", _vp), ("num_slots", _i64),
        ("output", _vp), ("output_state", _vp), ("chunk_states", _vp),
        ("chunk_indices", _vp), ("chunk_indices_dp", _vp), ("chunk_offsets", _vp),
        ("nt_pad", _i64), ("ntdp_pad", _i64),
        ("workspace", _vp), ("workspace_bytes", _sz),
        ("device_status", _vp),
        # input variants (ABI version 2)
        ("qkv_dtype", _int), ("g_dtype", _int), ("g_is_alpha", _int), ("beta_dtype", _int),
        ("initial_state_dtype", _int), ("num_q_heads", _int), ("num_k_heads", _int), ("num_v_heads", _int),
    ]


class GdpBackwardArgs(ctypes.Structure):
    """Mirror of ``gdp_backward_args``."""
    _fields_ = [
        ("fwd", ctypes.POINTER(GdpPrefillArgs)), ("d_output", _vp), ("d_final_state", _vp),
        ("dq", _vp), ("dk", _vp), ("dv", _vp), ("dg", _vp), ("dbeta", _vp), ("d_initial_state", _vp),
        ("workspace", _vp), ("workspace_bytes", _sz), ("device_status", _vp),
    ]


class GdpError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load_library(path: str | None = None):
    """Load libgdp_gb300.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(p)
    lib.gdp_prefill_varlen.restype = _int
    lib.gdp_prefill_varlen.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp]
    lib.gdp_prefill_varlen_profiled.restype = _int
    lib.gdp_prefill_varlen_profiled.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp, ctypes.POINTER(_vp), _int]
    lib.gdp_decode_step.restype = _int
    lib.gdp_decode_step.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp]
    lib.gdp_prefill_varlen_static_scratch.restype = _int
    lib.gdp_prefill_varlen_static_scratch.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp]
    lib.gdp_static_scratch_bytes.restype = _sz
    lib.gdp_arm_wait_expiry_test.restype = _int
    lib.gdp_arm_wait_expiry_test.argtypes = [ctypes.c_uint64]
    lib.gdp_debug_bounds_record.restype = _int
    lib.gdp_debug_bounds_record.argtypes = [ctypes.POINTER(_i64)]
    lib.gdp_arm_bounds_test.restype = _int
    lib.gdp_arm_bounds_test.argtypes = []
    lib.gdp_static_scratch_bytes.argtypes = []
    lib.gdp_prefill_varlen_backward.restype = _int
    lib.gdp_prefill_varlen_backward.argtypes = [ctypes.POINTER(GdpBackwardArgs), _vp]
    lib.gdp_backward_workspace_bytes.restype = _sz
    lib.gdp_backward_workspace_bytes.argtypes = [_i64, _i64, _int, _int, _int, _int]
    lib.gdp_prefill_workspace_bytes.restype = _sz
    lib.gdp_prefill_workspace_bytes.argtypes = [_i64, _i64, _int, _int, _int, _int]
    lib.gdp_prefill_transfer.restype = _int
    lib.gdp_prefill_transfer.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp, _vp]
    lib.gdp_chain_states.restype = _int
    lib.gdp_chain_states.argtypes = [_vp, _vp, _vp, _i64, _i64, _int, _int, _vp, _vp, _vp]
    lib.gdp_prefill_fused.restype = _int
    lib.gdp_prefill_fused.argtypes = [_i64, _i64, _int, _int, _int, _int] + [ctypes.POINTER(_i64)] * 3
    lib.gdp_prefill_varlen_fused.restype = _int
    lib.gdp_prefill_varlen_fused.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp]
    lib.gdp_prefill_varlen_fused_profiled.restype = _int
    lib.gdp_prefill_varlen_fused_profiled.argtypes = [ctypes.POINTER(GdpPrefillArgs), _vp, ctypes.POINTER(_vp), _int]
    lib.gdp_prefill_plan.restype = _int
    lib.gdp_prefill_plan.argtypes = [_i64, _i64, _int, _int, _int, _int] + [ctypes.POINTER(_i64)] * 4
    lib.gdp_build_descriptors.restype = _int
    lib.gdp_build_descriptors.argtypes = [_vp, _int, _i64, _i64, _int, _vp, _i64, _vp, _i64, _vp, _vp, _vp, _vp]
    lib.gdp_last_error.restype = ctypes.c_char_p
    lib.gdp_last_error.argtypes = []
    lib.gdp_abi_version.restype = _int
    lib.gdp_nt_pad.restype = _i64
    lib.gdp_nt_pad.argtypes = [_i64, _i64]
    lib.gdp_ntdp_pad.restype = _i64
    lib.gdp_ntdp_pad.argtypes = [_i64, _i64, _int]
    lib.gdp_prefill_args_size.restype = _sz
    if lib.gdp_prefill_args_size() != ctypes.sizeof(GdpPrefillArgs) or lib.gdp_abi_version() != GDP_ABI_VERSION:
        raise RuntimeError("gdp_prefill_args layout mismatch between the binding and the library")
    if path is None:
        _lib = lib
    return lib


# ---- the C entry points, same names ----------------------------------------------------------

def gdp_last_error() -> str:
    return load_library().gdp_last_error().decode()


def gdp_nt_pad(T: int, N: int) -> int:
    return int(load_library().gdp_nt_pad(T, N))


def gdp_ntdp_pad(T: int, N: int, M: int) -> int:
    return int(load_library().gdp_ntdp_pad(T, N, M))


def gdp_prefill_workspace_bytes(T: int, N: int, H: int, K: int, V: int, M: int) -> int:
    return int(load_library().gdp_prefill_workspace_bytes(T, N, H, K, V, M))


def gdp_prefill_plan(T: int, N: int, H: int, K: int, V: int, M: int) -> dict:
    """How a call of this shape runs: segments, piece_chunks (0 unless the chains are split),
    piece_rows and the number of kernel launches (shape-only)."""
    lib = load_library()
    out = [ctypes.c_int64() for _ in range(4)]
    st = lib.gdp_prefill_plan(T, N, H, K, V, M, *[ctypes.byref(x) for x in out])
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())
    return dict(zip(("segments", "piece_chunks", "piece_rows", "launches"), (int(x.value) for x in out)))


def gdp_prefill_fused(T: int, N: int, H: int, K: int, V: int, M: int):
    """The plan of gdp_prefill_varlen_fused for a common-contract call of this shape (dict with
    piece_chunks, piece_rows, launches), or None when it does not serve the shape."""
    out = [ctypes.c_int64() for _ in range(3)]
    ok = load_library().gdp_prefill_fused(T, N, H, K, V, M, *[ctypes.byref(x) for x in out])
    if not ok:
        return None
    return dict(zip(("piece_chunks", "piece_rows", "launches"), (int(x.value) for x in out)))


def gdp_prefill_varlen_fused(args: GdpPrefillArgs, stream: int | None = None) -> None:
    """Enqueue one prefill as the fused kernel (see the header) on ``stream``."""
    lib = load_library()
    st = lib.gdp_prefill_varlen_fused(ctypes.byref(args), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_prefill_varlen_fused_profiled(args: GdpPrefillArgs, events, stream: int | None = None) -> None:
    """As gdp_prefill_varlen_fused, recording the 4 torch.cuda.Event objects around the stages."""
    lib = load_library()
    handles = [e.cuda_event for e in events]
    if len(handles) != 4 or not all(handles):
        raise GdpError(GDP_ERR_INVALID_ARG, "need 4 created events (record each once before passing it)")
    arr = (_vp * 4)(*[ctypes.c_void_p(h) for h in handles])
    st = lib.gdp_prefill_varlen_fused_profiled(ctypes.byref(args), ctypes.c_void_p(_stream(stream)), arr, 4)
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def _stream(stream):
    return torch.cuda.current_stream().cuda_stream if stream is None else stream


def gdp_prefill_varlen(args: GdpPrefillArgs, stream: int | None = None) -> None:
    """Enqueue one prefill on ``stream`` (default: torch's current stream)."""
    lib = load_library()
    st = lib.gdp_prefill_varlen(ctypes.byref(args), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_prefill_varlen_profiled(args: GdpPrefillArgs, events, stream: int | None = None) -> None:
    """As gdp_prefill_varlen, recording the 4 torch.cuda.Event objects around the stages."""
    lib = load_library()
    handles = [e.cuda_event for e in events]
    if len(handles) != 4 or not all(handles):
        raise GdpError(GDP_ERR_INVALID_ARG, "need 4 created events (record each once before passing it)")
    arr = (_vp * 4)(*[ctypes.c_void_p(h) for h in handles])
    st = lib.gdp_prefill_varlen_profiled(ctypes.byref(args), ctypes.c_void_p(_stream(stream)), arr, len(events))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_static_scratch_bytes() -> int:
    """Size of the library's static scratch array (the largest workspace the
    static-scratch entry point serves)."""
    return int(load_library().gdp_static_scratch_bytes())


def gdp_arm_wait_expiry_test(limit_ns: int) -> None:
    """Arm the calling thread's next prefill call to exercise the bounded-wait failure path
    (its scan waits give up after limit_ns; one of them runs out); see the header."""
    lib = load_library()
    st = lib.gdp_arm_wait_expiry_test(int(limit_ns))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_debug_bounds_record() -> dict:
    """Debug-bounds builds: the range-check violations recorded since the last read (count, the
    first one's site, index and bound), then cleared; GdpError (UNSUPPORTED) in other builds."""
    lib = load_library()
    out = (_i64 * 4)()
    st = lib.gdp_debug_bounds_record(out)
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())
    return {"count": int(out[0]), "site": BOUNDS_SITES.get(int(out[1]), int(out[1])), "index": int(out[2]),
            "bound": int(out[3])}


def gdp_arm_bounds_test() -> None:
    """Debug-bounds builds: the calling thread's next prefill checks its output rows against T - 1
    (the last token's output stores fail their check and are skipped); see the header."""
    lib = load_library()
    st = lib.gdp_arm_bounds_test()
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_prefill_varlen_static_scratch(args: GdpPrefillArgs, stream: int | None = None) -> None:
    """The prefill without a caller workspace: the library's own static scratch
    (gdp_static_scratch_bytes()) is used instead, for callers that cannot allocate
    device memory; args.workspace is ignored.  Calls that overlap on the GPU race."""
    lib = load_library()
    st = lib.gdp_prefill_varlen_static_scratch(ctypes.byref(args), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_build_descriptors(cu_seqlens: torch.Tensor, T: int, num_householder: int, nt_pad: int | None = None,
                          ntdp_pad: int | None = None, device_status: torch.Tensor | None = None,
                          stream: int | None = None):
    """Device descriptors (chunk_indices [nt_pad,2], chunk_indices_dp [ntdp_pad,2], chunk_offsets [N+1])."""
    lib = load_library()
    N = cu_seqlens.numel() - 1
    nt_pad = gdp_nt_pad(T, N) if nt_pad is None else nt_pad
    ntdp_pad = gdp_ntdp_pad(T, N, num_householder) if ntdp_pad is None else ntdp_pad
    dev = cu_seqlens.device
    ci = torch.empty((nt_pad, 2), dtype=torch.int32, device=dev)
    cid = torch.empty((ntdp_pad, 2), dtype=torch.int32, device=dev)
    co = torch.empty(N + 1, dtype=torch.int32, device=dev)
    cod = torch.empty(N + 1, dtype=torch.int32, device=dev)
    st = lib.gdp_build_descriptors(
        _ptr(cu_seqlens), int(cu_seqlens.dtype == torch.int64), T, N, num_householder, _ptr(ci), nt_pad, _ptr(cid),
        ntdp_pad, _ptr(co), _ptr(cod), _ptr(device_status), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())
    return ci, cid, co


# ---- convenience wrapper ------------------------------------------------------------------------

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _addr(t):
    return t.data_ptr() if t is not None else None


def _set_variants(a, q, k, v, g, beta, initial_state, state, g_is_alpha):
    """Element types and head counts of the tensors -> the ABI-version-2 fields (the library
    checks the combinations)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in (torch.bfloat16, torch.float16) or t.dtype != q.dtype:
            raise GdpError(GDP_ERR_UNSUPPORTED, f"{name} must be bfloat16 or float16, like q (got {t.dtype})")
        if t.stride(-1) != 1:
            raise GdpError(GDP_ERR_INVALID_ARG, f"{name} must be contiguous in its last dimension")
    for name, t in (("g", g), ("beta", beta), ("initial_state", initial_state), ("state", state)):
        if t is not None and (t.dtype not in _DTYPE_CODE or not t.is_contiguous()):
            raise GdpError(GDP_ERR_UNSUPPORTED, f"{name} must be a contiguous float32/bfloat16/float16 tensor")
    if state is not None and state.dtype != torch.float32:
        raise GdpError(GDP_ERR_UNSUPPORTED, "the state cache is float32")
    a.qkv_dtype = _DTYPE_CODE[q.dtype]
    a.g_dtype = _DTYPE_CODE[g.dtype] if g is not None else 0
    a.g_is_alpha = int(bool(g_is_alpha))
    a.beta_dtype = _DTYPE_CODE[beta.dtype] if beta is not None else 0
    a.initial_state_dtype = _DTYPE_CODE[initial_state.dtype] if initial_state is not None else 0
    a.num_q_heads, a.num_k_heads, a.num_v_heads = q.shape[1], k.shape[1], v.shape[1]


def make_args(q, k, v, g, beta, cu_seqlens, num_householder, scale, initial_state, state, state_indices,
              output, output_state, chunk_states, chunk_indices, chunk_indices_dp, chunk_offsets,
              nt_pad, ntdp_pad, use_qk_l2norm, workspace, device_status, g_is_alpha=False) -> GdpPrefillArgs:
    """Fill a GdpPrefillArgs from tensors (no copies; the library checks shapes and modes).
    q [T,Hq,K], k [T*M,Hk,K], v [T*M,Hv,V]: H = max(Hq, Hv) state heads."""
    T, K = q.shape[0], q.shape[2]
    H = max(q.shape[1], v.shape[1])
    V = v.shape[-1]
    a = GdpPrefillArgs()
    _set_variants(a, q, k, v, g, beta, initial_state, state, g_is_alpha)
    a.q, a.q_stride_t, a.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    a.k, a.k_stride_t, a.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    a.v, a.v_stride_t, a.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
    a.g, a.beta = _addr(g), _addr(beta)
    a.cu_seqlens = cu_seqlens.data_ptr()
    a.cu_seqlens_int64 = int(cu_seqlens.dtype == torch.int64)
    a.T, a.N = T, cu_seqlens.numel() - 1
    a.H, a.K, a.V, a.num_householder = H, K, V, int(num_householder)
    a.scale = 0.0 if scale is None else float(scale)
    a.use_qk_l2norm = int(bool(use_qk_l2norm))
    a.initial_state, a.state, a.state_indices = _addr(initial_state), _addr(state), _addr(state_indices)
    a.num_slots = state.shape[0] if state is not None else 0
    a.output, a.output_state, a.chunk_states = _addr(output), _addr(output_state), _addr(chunk_states)
    a.chunk_indices, a.chunk_indices_dp, a.chunk_offsets = _addr(chunk_indices), _addr(chunk_indices_dp), _addr(
        chunk_offsets)
    a.nt_pad = int(nt_pad or 0)
    a.ntdp_pad = int(ntdp_pad or 0)
    a.workspace = _addr(workspace)
    a.workspace_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    a.device_status = _addr(device_status)
    return a


def gdp_backward_workspace_bytes(T: int, N: int, H: int, K: int, V: int, M: int) -> int:
    return int(load_library().gdp_backward_workspace_bytes(T, N, H, K, V, M))


def gdp_prefill_varlen_backward(args: GdpBackwardArgs, stream: int | None = None) -> None:
    """Enqueue the backward pass on ``stream`` (default: torch's current stream).  The
    forward arguments ``args.fwd`` must stay alive during the call."""
    lib = load_library()
    st = lib.gdp_prefill_varlen_backward(ctypes.byref(args), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def backward_args(fwd: GdpPrefillArgs, d_output, d_final_state, dq, dk, dv, dg, dbeta, d_initial_state, workspace,
                  device_status=None) -> GdpBackwardArgs:
    """Fill a GdpBackwardArgs from tensors (no copies); keep ``fwd`` alive while it is used."""
    b = GdpBackwardArgs()
    b.fwd = ctypes.pointer(fwd)
    b.d_output, b.d_final_state = _addr(d_output), _addr(d_final_state)
    b.dq, b.dk, b.dv, b.dg, b.dbeta = _addr(dq), _addr(dk), _addr(dv), _addr(dg), _addr(dbeta)
    b.d_initial_state = _addr(d_initial_state)
    b.workspace = workspace.data_ptr()
    b.workspace_bytes = workspace.numel() * workspace.element_size()
    b.device_status = _addr(device_status)
    return b


def chunk_gated_delta_product_backward(q, k, v, g, beta, cu_seqlens, num_householder, d_output, scale=None,
                                       initial_state=None, d_final_state=None, use_qk_l2norm_in_kernel=False,
                                       workspace=None, device_status=None, stream=None):
    """Gradients of the prefill for a loss with dL/do = ``d_output`` [T,H,V] (bf16) and
    dL/dS_final = ``d_final_state`` [N,H,V,K] (fp32, or None).  q [T,H,K], k [T*M,H,K],
    v [T*M,H,V] bf16; g [T,H] natural-log decay fp32 (or None); beta [T*M,H] fp32 (or None);
    initial_state [N,H,V,K] fp32 (or None).  Returns a dict of fp32 tensors dq, dk, dv, dg
    (None without g), dbeta and d_initial_state (None without an initial state)."""
    T, H, K = q.shape
    V = v.shape[-1]
    M = int(num_householder)
    N = cu_seqlens.numel() - 1
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    out = {"dq": torch.empty((T, H, K), **f32), "dk": torch.empty((T * M, H, K), **f32),
           "dv": torch.empty((T * M, H, V), **f32),
           "dg": torch.empty((T, H), **f32) if g is not None else None,
           "dbeta": torch.empty((T * M, H), **f32),
           "d_initial_state": torch.empty((N, H, V, K), **f32) if initial_state is not None else None}
    if workspace is None:
        nbytes = gdp_backward_workspace_bytes(T, N, H, K, V, M)
        if nbytes == 0:
            raise GdpError(GDP_ERR_INVALID_ARG, "invalid shape for the workspace query")
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    fa = make_args(q, k, v, g, beta, cu_seqlens, M, scale, initial_state, None, None, None, None, None, None, None,
                   None, None, None, use_qk_l2norm_in_kernel, None, None)
    b = backward_args(fa, d_output, d_final_state, out["dq"], out["dk"], out["dv"], out["dg"], out["dbeta"],
                      out["d_initial_state"], workspace, device_status)
    gdp_prefill_varlen_backward(b, stream)
    return out


def gdp_decode_step(args: GdpPrefillArgs, stream: int | None = None) -> None:
    """Enqueue one decode step (one token per sequence, T == N) on ``stream``."""
    lib = load_library()
    st = lib.gdp_decode_step(ctypes.byref(args), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def decode_args(q, k, v, g, beta, num_householder, scale, initial_state, state, state_indices, output,
                output_state, use_qk_l2norm, device_status, g_is_alpha=False) -> GdpPrefillArgs:
    """GdpPrefillArgs of a decode step: q [N,Hq,K], k/v [N*M,Hk|Hv,K|V] bf16 or f16 (no copies)."""
    N, K = q.shape[0], q.shape[2]
    H = max(q.shape[1], v.shape[1])
    V = v.shape[-1]
    a = GdpPrefillArgs()
    _set_variants(a, q, k, v, g, beta, initial_state, state, g_is_alpha)
    a.q, a.q_stride_t, a.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    a.k, a.k_stride_t, a.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    a.v, a.v_stride_t, a.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
    a.g, a.beta = _addr(g), _addr(beta)
    a.T, a.N = N, N
    a.H, a.K, a.V, a.num_householder = H, K, V, int(num_householder)
    a.scale = 0.0 if scale is None else float(scale)
    a.use_qk_l2norm = int(bool(use_qk_l2norm))
    a.initial_state, a.state, a.state_indices = _addr(initial_state), _addr(state), _addr(state_indices)
    a.num_slots = state.shape[0] if state is not None else 0
    a.output, a.output_state = output.data_ptr(), _addr(output_state)
    a.device_status = _addr(device_status)
    return a


def gated_delta_product_decode(q, k, v, g=None, beta=None, num_householder=1, scale=None, initial_state=None,
                               output_final_state=False, use_qk_l2norm_in_kernel=False, state=None,
                               state_indices=None, output=None, output_state=None, device_status=None,
                               stream=None, g_is_alpha=False):
    """One decode step: token i of sequence i, q [N,Hq,K], k/v [N*M,Hk|Hv,...] bf16 or f16,
    g [N,H] (natural-log decay, or alpha itself when ``g_is_alpha``), beta [N*M,H]; H = max(Hq, Hv).

    Returns ``o`` [N,H,V] in q's dtype, or ``(o, final_state)`` when output_final_state (dense
    mode).  In state-cache mode the cache is updated in place at ``state_indices``.
    """
    N, K = q.shape[0], q.shape[2]
    H = max(q.shape[1], v.shape[1])
    V = v.shape[-1]
    if output is None:
        output = torch.empty((N, H, V), dtype=q.dtype, device=q.device)
    if output_final_state and state is None and output_state is None:
        output_state = torch.empty((N, H, V, K), dtype=torch.float32, device=q.device)
    a = decode_args(q, k, v, g, beta, num_householder, scale, initial_state, state, state_indices, output,
                    output_state, use_qk_l2norm_in_kernel, device_status, g_is_alpha)
    gdp_decode_step(a, stream)
    if output_final_state and state is None:
        return output, output_state
    return output


def alloc_workspace(T, N, H, K, V, M, device) -> torch.Tensor:
    nbytes = gdp_prefill_workspace_bytes(T, N, H, K, V, M)
    if nbytes == 0:
        raise GdpError(GDP_ERR_INVALID_ARG, "invalid shape for the workspace query")
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def chunk_gated_delta_product(q, k, v, g=None, beta=None, cu_seqlens=None, num_householder=1, scale=None,
                              initial_state=None, output_final_state=False, use_qk_l2norm_in_kernel=False,
                              chunk_indices=None, chunk_indices_dp=None, chunk_offsets=None, state=None,
                              state_indices=None, return_chunk_states=False, output=None, output_state=None,
                              workspace=None, device_status=None, nt_pad=None, ntdp_pad=None, stream=None,
                              g_is_alpha=False, fused=False):
    """Chunked Gated DeltaProduct varlen prefill on the GPU (``fused``: through
    gdp_prefill_varlen_fused instead of gdp_prefill_varlen).

    q [T,Hq,K] (or [1,T,Hq,K]), k/v [T*M,Hk,K]/[T*M,Hv,V] bf16 or float16 (one type);
    H = max(Hq, Hv) state heads, Hk equal to Hq or Hv, each dividing H.  g [T,H]
    natural-log decays (or alpha itself in linear space when ``g_is_alpha``), fp32,
    bf16 or f16; beta [T*M,H] fp32 or q's dtype; initial_state [N,H,V,K] fp32 or bf16;
    cu_seqlens [N+1] int32/int64 (required).  Returns ``o`` [T,H,V] in q's dtype, or
    ``(o, final_state)`` when output_final_state, or ``(o, final_state, chunk_states)``
    when return_chunk_states (both fp32).  In state-cache mode (``state``/``state_indices``)
    the final state is written into the cache and ``final_state`` is None.
    """
    if cu_seqlens is None:
        raise GdpError(GDP_ERR_INVALID_ARG, "cu_seqlens is required (packed THD input only)")
    if q.dim() == 4 and q.shape[0] == 1:
        q, k, v = q[0], k[0], v[0]
    if g is not None and g.dim() == 3:
        g = g[0]
    if beta is not None and beta.dim() == 3:
        beta = beta[0]
    T, K = q.shape[0], q.shape[2]
    H = max(q.shape[1], v.shape[1])
    V = v.shape[-1]
    M = int(num_householder)
    N = cu_seqlens.numel() - 1
    dev = q.device
    if output is None:
        output = torch.empty((T, H, V), dtype=q.dtype, device=dev)
    if output_final_state and state is None and output_state is None:
        output_state = torch.empty((N, H, V, K), dtype=torch.float32, device=dev)
    cs = None
    if return_chunk_states:
        rows = nt_pad if nt_pad else gdp_nt_pad(T, N)
        cs = torch.zeros((rows, H, V, K), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(T, N, H, K, V, M, dev)
    a = make_args(q, k, v, g, beta, cu_seqlens, M, scale, initial_state, state, state_indices, output,
                  output_state if state is None else None, cs, chunk_indices, chunk_indices_dp, chunk_offsets,
                  nt_pad, ntdp_pad, use_qk_l2norm_in_kernel, workspace, device_status, g_is_alpha)
    (gdp_prefill_varlen_fused if fused else gdp_prefill_varlen)(a, stream)
    final = output_state if (output_final_state and state is None) else None
    if return_chunk_states:
        return output, final, cs
    if output_final_state:
        return output, final
    return output


# ---- sequence-sharded prefill by state passing ----------------------------------------------

def gdp_prefill_transfer(args: GdpPrefillArgs, pairs: int, stream: int | None = None) -> None:
    """Enqueue the transfer pairs (B, Phi) of every sequence of ``args`` into ``pairs``."""
    lib = load_library()
    st = lib.gdp_prefill_transfer(ctypes.byref(args), ctypes.c_void_p(pairs), ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def gdp_chain_states(s0, phi, b, steps: int, N: int, H: int, d: int, s_out, device_status=None,
                     stream: int | None = None) -> None:
    """Enqueue S_{j+1} = S_j Phi_j + B_j (j < steps) from S_0 = s0 (None: zero) into s_out."""
    lib = load_library()
    st = lib.gdp_chain_states(_ptr(s0), _ptr(phi), _ptr(b), steps, N, H, d, _ptr(s_out), _ptr(device_status),
                              ctypes.c_void_p(_stream(stream)))
    if st != GDP_OK:
        raise GdpError(st, lib.gdp_last_error().decode())


def chunk_gated_delta_product_transfer(q, k, v, g=None, beta=None, cu_seqlens=None, num_householder=1, scale=None,
                                       use_qk_l2norm_in_kernel=False, workspace=None, device_status=None,
                                       stream=None, g_is_alpha=False):
    """The transfer pairs of a shard: returns ``pairs`` [2, N, H, V, K] fp32 with pairs[0] = B (the
    state after each sequence from a zero state) and pairs[1] = Phi (from the identity with v = 0),
    so that the final state from any initial state S_0 is S_0 @ Phi + B.  Inputs as for
    chunk_gated_delta_product."""
    if cu_seqlens is None:
        raise GdpError(GDP_ERR_INVALID_ARG, "cu_seqlens is required (packed THD input only)")
    T, K = q.shape[0], q.shape[2]
    H = max(q.shape[1], v.shape[1])
    V = v.shape[-1]
    M = int(num_householder)
    N = cu_seqlens.numel() - 1
    pairs = torch.empty((2, N, H, V, K), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(T, N, H, K, V, M, q.device)
    a = make_args(q, k, v, g, beta, cu_seqlens, M, scale, None, None, None, None, None, None, None, None, None,
                  None, None, use_qk_l2norm_in_kernel, workspace, device_status, g_is_alpha)
    gdp_prefill_transfer(a, pairs.data_ptr(), stream)
    return pairs


def chain_states(s0, phi, b, device_status=None, stream=None):
    """S_out [steps+1, N, H, d, d] with S_out[0] = s0 (None: zero), S_out[j+1] = S_out[j] @ phi[j] + b[j]."""
    steps, N, H, d = phi.shape[0], phi.shape[1], phi.shape[2], phi.shape[-1]
    for x in (phi, b) + ((s0,) if s0 is not None else ()):
        if x.dtype != torch.float32 or not x.is_contiguous():
            raise GdpError(GDP_ERR_INVALID_ARG, "chain_states takes contiguous fp32 tensors")
    s_out = torch.empty((steps + 1, N, H, d, d), dtype=torch.float32, device=phi.device)
    gdp_chain_states(s0, phi, b, steps, N, H, d, s_out, device_status, stream)
    return s_out


def gather_transfer_pairs(pairs, group=None):
    """All ranks' transfer pairs in rank order: [R, 2, N, H, V, K] (the one exchange of the
    sequence-sharded prefill; any torch.distributed backend)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = [torch.empty_like(pairs) for _ in range(world)]
    dist.all_gather(out, pairs.contiguous(), group=group)
    return torch.stack(out)


def sequence_parallel_steps(transfer, chain, run, initial_state, group=None):
    """The host logic of the sequence-sharded prefill over its three device steps:
    ``transfer()`` gives this rank's pairs [2, N, H, V, K], the pairs of all ranks are
    all-gathered, ``chain(s0, phi, b)`` ([steps + 1, ...]) chains those of the ranks before this
    one onto ``initial_state``, and ``run(s_in)`` runs the shard from the result."""
    import torch.distributed as dist
    rank = dist.get_rank(group)
    allp = gather_transfer_pairs(transfer(), group)  # [R, 2, N, H, V, K]
    if rank == 0:
        return run(initial_state)
    s0 = None if initial_state is None else initial_state.to(torch.float32).contiguous()
    return run(chain(s0, allp[:rank, 1].contiguous(), allp[:rank, 0].contiguous())[rank])


def chunk_gated_delta_product_sequence_parallel(q, k, v, g=None, beta=None, cu_seqlens=None, num_householder=1,
                                                scale=None, initial_state=None, use_qk_l2norm_in_kernel=False,
                                                return_chunk_states=False, group=None, g_is_alpha=False):
    """Prefill of sequences whose tokens are split over the ranks of ``group`` in rank order:
    this rank holds every sequence's shard r (consecutive whole tokens; empty shards allowed),
    packed with its own ``cu_seqlens``.  ``initial_state`` [N, H, V, K] is the state before
    shard 0 (the same on every rank, or None).  Each rank computes its shard's transfer pairs on
    the GPU, the pairs are all-gathered (the one exchange), each rank chains the pairs of the ranks
    before it onto the initial state (GPU) and runs its shard from there (GPU).  Returns
    ``(o, final_state)`` (``chunk_states`` third when asked): final_state is the state after this
    rank's shard, the sequence's final state on the last rank; chunk-state rows are per shard."""
    def transfer():
        return chunk_gated_delta_product_transfer(q, k, v, g, beta, cu_seqlens, num_householder, scale,
                                                  use_qk_l2norm_in_kernel, g_is_alpha=g_is_alpha)

    def run(s_in):
        return chunk_gated_delta_product(q, k, v, g, beta, cu_seqlens, num_householder, scale, initial_state=s_in,
                                         output_final_state=True, use_qk_l2norm_in_kernel=use_qk_l2norm_in_kernel,
                                         return_chunk_states=return_chunk_states, g_is_alpha=g_is_alpha)

    return sequence_parallel_steps(transfer, chain_states, run, initial_state, group)
