"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point the header declares, agrees with the binding on the argument
struct, answers the shape-only queries, and rejects bad arguments before any
launch with the documented status codes."""
import ctypes
import os
import re

import pytest

import chunked_gated_deltaproduct_gb300 as pkg
from chunked_gated_deltaproduct_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return pkg.load_library()


def _declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"\b(gdp_[a-z0-9_]+)\s*\(", text):
            names.add(m.group(1))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    declared = _declared_functions()
    assert "gdp_prefill_varlen" in declared and "gdp_build_descriptors" in declared
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert lib.gdp_abi_version() == pkg.GDP_ABI_VERSION == 2


def test_debug_bounds_build_exports_and_normal_build_declines(lib):
    """The debug-bounds variant builds and exports the same symbols; in the normal build its two
    entry points return GDP_ERR_UNSUPPORTED without touching the device."""
    from chunked_gated_deltaproduct_gb300 import binding, build as libbuild

    path = libbuild.build(debug_bounds=True)
    dbg = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(dbg, name), f"{name} missing from the debug-bounds build"
    for fn in (pkg.gdp_debug_bounds_record, pkg.gdp_arm_bounds_test):
        with pytest.raises(pkg.GdpError) as e:
            fn()
        assert e.value.status == pkg.GDP_ERR_UNSUPPORTED
    assert binding.DEBUG_LIB_PATH == path


def test_args_struct_layout(lib):
    assert lib.gdp_prefill_args_size() == ctypes.sizeof(pkg.GdpPrefillArgs)


def test_padding_bounds_and_workspace(lib):
    assert pkg.gdp_nt_pad(1421, 4) == 26 and pkg.gdp_ntdp_pad(1421, 4, 2) == 48
    assert pkg.gdp_ntdp_pad(257, 1, 3) == 13
    a = pkg.gdp_prefill_workspace_bytes(65536, 1, 32, 128, 128, 2)
    b = pkg.gdp_prefill_workspace_bytes(65536, 1, 32, 128, 128, 2)
    assert a == b > 0 and a % 256 == 0
    assert pkg.gdp_prefill_workspace_bytes(-1, 1, 1, 64, 64, 1) == 0
    assert pkg.gdp_prefill_workspace_bytes(10, 1, 1, 64, 64, 0) == 0


def _args(**over):
    a = pkg.GdpPrefillArgs()
    T, N, H, K = 8, 1, 1, 64
    fake = 1 << 20  # a 16-byte aligned non-NULL address; never dereferenced on these paths
    a.q = a.k = a.v = a.output = fake
    a.q_stride_t, a.q_stride_h = H * K, K
    a.k_stride_t, a.k_stride_h = H * K, K
    a.v_stride_t, a.v_stride_h = H * K, K
    a.cu_seqlens = fake
    a.T, a.N, a.H, a.K, a.V, a.num_householder = T, N, H, K, K, 1
    a.workspace = fake
    a.workspace_bytes = pkg.gdp_prefill_workspace_bytes(T, N, H, K, K, 1)
    for k, v in over.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("over,status", [
    (dict(K=96, V=96), pkg.GDP_ERR_UNSUPPORTED),
    (dict(K=64, V=128), pkg.GDP_ERR_UNSUPPORTED),
    (dict(num_householder=0), pkg.GDP_ERR_INVALID_ARG),
    (dict(q=None), pkg.GDP_ERR_INVALID_ARG),
    (dict(q_stride_h=60), pkg.GDP_ERR_INVALID_ARG),
    (dict(q=(1 << 20) + 8), pkg.GDP_ERR_INVALID_ARG),
    (dict(initial_state=1 << 21, state=1 << 22, state_indices=1 << 23, num_slots=4), pkg.GDP_ERR_INVALID_ARG),
    (dict(state=1 << 22), pkg.GDP_ERR_INVALID_ARG),
    (dict(initial_state=(1 << 21) + 4), pkg.GDP_ERR_INVALID_ARG),
    (dict(chunk_states=(1 << 21) + 8), pkg.GDP_ERR_INVALID_ARG),
    (dict(state=1 << 22, state_indices=1 << 23, num_slots=4, output_state=1 << 24), pkg.GDP_ERR_INVALID_ARG),
    (dict(initial_state=1 << 24, output_state=(1 << 24) + 4096), pkg.GDP_ERR_ALIAS),
    (dict(chunk_indices=1 << 21), pkg.GDP_ERR_INVALID_ARG),
    (dict(T=1 << 22, H=4096, q_stride_t=4096 * 64, k_stride_t=4096 * 64, v_stride_t=4096 * 64),
     pkg.GDP_ERR_UNSUPPORTED),  # chunk-state rows beyond 32-bit tensor coordinates
    (dict(workspace=None), pkg.GDP_ERR_WORKSPACE),
    (dict(workspace=(1 << 20) + 16), pkg.GDP_ERR_WORKSPACE),
    (dict(workspace_bytes=64), pkg.GDP_ERR_WORKSPACE),
    (dict(T=200, nt_pad=1, ntdp_pad=1, chunk_indices=1 << 21, chunk_indices_dp=1 << 21, chunk_offsets=1 << 21),
     pkg.GDP_ERR_INVALID_ARG),
    # input variants (ABI version 2)
    (dict(qkv_dtype=pkg.GDP_DTYPE_F32), pkg.GDP_ERR_UNSUPPORTED),
    (dict(qkv_dtype=7), pkg.GDP_ERR_UNSUPPORTED),
    (dict(g_dtype=9), pkg.GDP_ERR_UNSUPPORTED),
    (dict(beta_dtype=pkg.GDP_DTYPE_F16), pkg.GDP_ERR_UNSUPPORTED),  # neither fp32 nor the (bf16) q type
    (dict(qkv_dtype=pkg.GDP_DTYPE_F16, beta_dtype=pkg.GDP_DTYPE_BF16), pkg.GDP_ERR_UNSUPPORTED),
    (dict(initial_state_dtype=pkg.GDP_DTYPE_F16), pkg.GDP_ERR_UNSUPPORTED),
    (dict(g_is_alpha=2), pkg.GDP_ERR_INVALID_ARG),
    (dict(H=4, num_q_heads=3, num_k_heads=3), pkg.GDP_ERR_INVALID_ARG),  # 3 does not divide 4
    (dict(H=4, num_q_heads=2, num_k_heads=2, num_v_heads=2), pkg.GDP_ERR_INVALID_ARG),  # H != max(q, v)
    (dict(H=4, num_q_heads=4, num_k_heads=1, num_v_heads=2), pkg.GDP_ERR_INVALID_ARG),  # k neither q nor v
    (dict(H=4, num_q_heads=2, num_k_heads=2, num_v_heads=4, q_stride_t=64, k_stride_t=128, v_stride_t=256),
     pkg.GDP_ERR_INVALID_ARG),  # q rows of 2 heads need a stride of 128
    (dict(initial_state=1 << 24, initial_state_dtype=pkg.GDP_DTYPE_BF16, output_state=(1 << 24) + 4096),
     pkg.GDP_ERR_ALIAS),  # the bf16 state spans 8 KB
])
def test_host_validation(lib, over, status):
    a = _args(**over)
    st = lib.gdp_prefill_varlen(ctypes.byref(a), None)
    assert st == status, (st, pkg.gdp_last_error())
    assert pkg.gdp_last_error() != ""


def test_profiled_needs_four_events(lib):
    a = _args()
    st = lib.gdp_prefill_varlen_profiled(ctypes.byref(a), None, None, 0)
    assert st == pkg.GDP_ERR_INVALID_ARG


def test_empty_batch_is_ok_without_launch(lib):
    a = _args(T=0, N=0)
    a.workspace_bytes = pkg.gdp_prefill_workspace_bytes(0, 0, 1, 64, 64, 1)
    assert lib.gdp_prefill_varlen(ctypes.byref(a), None) == pkg.GDP_OK
    assert pkg.gdp_last_error() == ""


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError):
        pkg.load_library(str(tmp_path / "nope.so"))


@pytest.mark.parametrize("over,status", [
    (dict(qkv_dtype=pkg.GDP_DTYPE_F32), pkg.GDP_ERR_UNSUPPORTED),
    (dict(H=4, num_q_heads=3, num_k_heads=3), pkg.GDP_ERR_INVALID_ARG),
    (dict(g_is_alpha=-1), pkg.GDP_ERR_INVALID_ARG),
    # an exact in-place update exists only for an fp32 initial state
    (dict(initial_state=1 << 24, output_state=1 << 24, initial_state_dtype=pkg.GDP_DTYPE_BF16), pkg.GDP_ERR_ALIAS),
])
def test_decode_host_validation(lib, over, status):
    a = _args(T=1, N=1, **over)
    st = lib.gdp_decode_step(ctypes.byref(a), None)
    assert st == status, (st, pkg.gdp_last_error())
    assert pkg.gdp_last_error() != ""


def _bwd(lib, fwd_over=None, **over):
    a = _args(**(fwd_over or {}))
    fake = 1 << 20
    b = pkg.GdpBackwardArgs()
    b.fwd = ctypes.pointer(a)
    b.d_output = b.dq = b.dk = b.dv = fake
    b.workspace = fake
    b.workspace_bytes = pkg.gdp_backward_workspace_bytes(a.T, a.N, a.H, a.K, a.V, a.num_householder)
    for k, v in over.items():
        setattr(b, k, v)
    return lib.gdp_prefill_varlen_backward(ctypes.byref(b), None), a


@pytest.mark.parametrize("fwd_over,over,status", [
    (dict(qkv_dtype=pkg.GDP_DTYPE_F16), {}, pkg.GDP_ERR_UNSUPPORTED),
    (dict(g_is_alpha=1), {}, pkg.GDP_ERR_UNSUPPORTED),
    (dict(g_dtype=pkg.GDP_DTYPE_BF16), {}, pkg.GDP_ERR_UNSUPPORTED),
    (dict(initial_state_dtype=pkg.GDP_DTYPE_BF16), {}, pkg.GDP_ERR_UNSUPPORTED),
    (dict(H=4, num_q_heads=2, num_k_heads=2, num_v_heads=4), {}, pkg.GDP_ERR_UNSUPPORTED),
    (dict(state=1 << 22, state_indices=1 << 23, num_slots=4), {}, pkg.GDP_ERR_UNSUPPORTED),
    (dict(K=96, V=96), {}, pkg.GDP_ERR_UNSUPPORTED),
    ({}, dict(d_output=None), pkg.GDP_ERR_INVALID_ARG),
    ({}, dict(dk=None), pkg.GDP_ERR_INVALID_ARG),
    ({}, dict(dq=(1 << 20) + 4), pkg.GDP_ERR_INVALID_ARG),
    ({}, dict(workspace_bytes=64), pkg.GDP_ERR_WORKSPACE),
    ({}, dict(workspace=None), pkg.GDP_ERR_WORKSPACE),
])
def test_backward_host_validation(lib, fwd_over, over, status):
    st, _ = _bwd(lib, fwd_over, **over)
    assert st == status, (st, pkg.gdp_last_error())
    assert pkg.gdp_last_error() != ""


def test_backward_null_forward_args(lib):
    b = pkg.GdpBackwardArgs()
    assert lib.gdp_prefill_varlen_backward(ctypes.byref(b), None) == pkg.GDP_ERR_INVALID_ARG


def test_backward_workspace_covers_forward():
    for shape in [(1421, 4, 8, 128, 128, 2), (65536, 1, 32, 128, 128, 2), (256, 1, 2, 64, 64, 1)]:
        assert pkg.gdp_backward_workspace_bytes(*shape) > pkg.gdp_prefill_workspace_bytes(*shape) > 0
    assert pkg.gdp_backward_workspace_bytes(10, 1, 1, 64, 64, 0) == 0


def test_prefill_plan(lib):
    """The shape-only plan: plain, segmented or split chains, and the launches each enqueues."""
    plain = pkg.gdp_prefill_plan(256, 1, 2, 64, 64, 1)  # four chunks: nothing to split
    assert plain == {"segments": 1, "piece_chunks": 0, "piece_rows": 0, "launches": 3}
    split = pkg.gdp_prefill_plan(1421, 4, 8, 64, 64, 2)
    # 4 sequences x 8 heads at head size 64: the staged kernels, split chains
    assert split["segments"] == 1 and split["piece_chunks"] == 6 and split["launches"] == 5
    assert split["piece_rows"] * 8 <= 128
    assert pkg.gdp_prefill_plan(32768, 8, 16, 128, 128, 3)["piece_chunks"] == 0  # 128 chains fill the GPU
    seg = pkg.gdp_prefill_plan(65536, 1, 32, 128, 128, 2)
    assert seg["segments"] == 16 and seg["piece_chunks"] == 0 and seg["launches"] == 33
    # gdp_prefill_varlen_fused's plan: one long chain per head splits into pieces (descriptors,
    # pass 1, combine, pass 2); many chains run whole (descriptors + the fused kernel)
    fused = pkg.gdp_prefill_fused(65536, 1, 32, 128, 128, 2)
    assert fused == {"piece_chunks": 683, "piece_rows": 4, "launches": 4}
    assert pkg.gdp_prefill_fused(32768, 8, 16, 128, 128, 3) == {"piece_chunks": 0, "piece_rows": 0, "launches": 2}
    assert pkg.gdp_prefill_fused(1421, 4, 8, 128, 128, 2)["piece_chunks"] == 6
    assert pkg.gdp_prefill_fused(65536, 1, 32, 128, 128, 1) is None  # M = 1: its tensor memory does not fit
    assert pkg.gdp_prefill_fused(4096, 2, 2, 64, 64, 2) is None  # head size 64
    assert pkg.gdp_prefill_plan(5000, 33, 1, 64, 64, 2)["piece_chunks"] == 0  # more than 32 sequences
    assert pkg.gdp_prefill_plan(0, 0, 4, 64, 64, 2)["launches"] == 0
    with pytest.raises(pkg.GdpError):
        pkg.gdp_prefill_plan(10, 1, 1, 64, 64, 0)
    # a split call needs workspace for the pieces' B, Phi and entering states
    assert (pkg.gdp_prefill_workspace_bytes(1421, 4, 8, 64, 64, 2)
            >= 3 * split["piece_rows"] * 8 * 64 * 64 * 4)
    assert (pkg.gdp_prefill_workspace_bytes(65536, 1, 32, 128, 128, 2)
            >= 3 * fused["piece_rows"] * 32 * 128 * 128 * 4)  # the fused entry point's pieces


@pytest.mark.parametrize("T,N,H,M", [(1421, 4, 8, 2), (3000, 1, 1, 1), (1143, 4, 2, 3), (5000, 32, 1, 2),
                                     (700, 3, 4, 4)])
def test_piece_rows_bound_every_length_mix(lib, T, N, H, M):
    """The kernels number pieces row by row up to piece_rows: for any split of T tokens over N
    sequences, sum_i max(1, ceil(ceil(L_i M / 64) / len)) stays within that bound."""
    import numpy as np
    plan = pkg.gdp_prefill_plan(T, N, H, 64, 64, M)
    ln, rows = plan["piece_chunks"], plan["piece_rows"]
    assert ln > 0 and rows * H <= 128
    rng = np.random.default_rng(T + N)
    mixes = [np.full(N, T // N) + (np.arange(N) < T % N), np.eye(N, dtype=int)[0] * T]
    for _ in range(200):
        cuts = np.sort(rng.integers(0, T + 1, N - 1))
        mixes.append(np.diff(np.concatenate([[0], cuts, [T]])))
    for L in mixes:
        assert L.sum() == T and (L >= 0).all()
        pieces = sum(max(1, -(-(-(-int(x) * M // 64)) // ln)) for x in L)
        assert pieces <= rows, (list(L), pieces, rows)


def test_transfer_and_chain_host_validation(lib):
    """The sequence-sharded prefill's entry points reject bad arguments before any launch."""
    vp = ctypes.c_void_p
    assert lib.gdp_prefill_transfer(None, None, None) == pkg.GDP_ERR_INVALID_ARG
    a = _args()
    assert lib.gdp_prefill_transfer(ctypes.byref(a), None, None) == pkg.GDP_ERR_INVALID_ARG  # pairs missing
    assert lib.gdp_prefill_transfer(ctypes.byref(a), vp(0x1008), None) == pkg.GDP_ERR_INVALID_ARG  # misaligned
    ch = lib.gdp_chain_states
    assert ch(None, None, None, 1, 1, 1, 96, vp(0x1000), None, None) == pkg.GDP_ERR_INVALID_ARG  # d not 64 / 128
    assert ch(None, None, None, -1, 1, 1, 64, vp(0x1000), None, None) == pkg.GDP_ERR_INVALID_ARG
    assert ch(None, None, None, 2, 1, 1, 64, vp(0x1000), None, None) == pkg.GDP_ERR_INVALID_ARG  # phi, b missing
    assert ch(None, None, None, 0, 1, 1, 64, None, None, None) == pkg.GDP_ERR_INVALID_ARG  # s_out missing
    assert ch(vp(0x1004), None, None, 0, 1, 1, 64, vp(0x2000), None, None) == pkg.GDP_ERR_INVALID_ARG
    assert ch(vp(0x1000), None, None, 0, 1, 1, 64, vp(0x1000), None, None) == pkg.GDP_ERR_ALIAS
    assert ch(None, vp(0x10000), vp(0x20000), 1, 1, 1, 64, vp(0x20000 + 4096), None, None) == pkg.GDP_ERR_ALIAS
    assert ch(None, None, None, 0, 0, 1, 64, None, None, None) == pkg.GDP_OK  # N = 0: nothing to do
    empty = _args(N=0, T=0)
    assert lib.gdp_prefill_transfer(ctypes.byref(empty), None, None) == pkg.GDP_OK  # no sequences, no launch
    assert lib.gdp_prefill_transfer(ctypes.byref(_args(K=96, V=96)), vp(0x1000), None) == pkg.GDP_ERR_UNSUPPORTED


def test_sequence_parallel_wrappers_reject_bad_tensors():
    """The binding's checks that run before any library call."""
    import torch
    with pytest.raises(pkg.GdpError):
        pkg.chain_states(None, torch.zeros((1, 1, 1, 64, 64), dtype=torch.float16), torch.zeros((1, 1, 1, 64, 64)))
    with pytest.raises(pkg.GdpError):
        pkg.chain_states(None, torch.zeros((1, 1, 1, 64, 64)).transpose(-1, -2), torch.zeros((1, 1, 1, 64, 64)))
    with pytest.raises(pkg.GdpError):
        q = torch.zeros((4, 1, 64), dtype=torch.bfloat16)
        pkg.chunk_gated_delta_product_transfer(q, q, q, cu_seqlens=None)


def test_static_scratch_size_matches_header(lib):
    """The static-scratch size the library reports is the header's GDP_STATIC_SCRATCH_BYTES."""
    text = open(os.path.join(HEADER_DIR, "gdp_prefill.h")).read()
    m = re.search(r"#define\s+GDP_STATIC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", text)
    assert m, "GDP_STATIC_SCRATCH_BYTES not found in the header"
    assert pkg.gdp_static_scratch_bytes() == int(m.group(1)) << int(m.group(2))
