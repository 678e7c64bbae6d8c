"""GB300-native (sm_103a) chunked Gated DeltaProduct varlen prefill.

The computation lives in ``libgdp_gb300.so`` (hand-written CUDA, C ABI in
``include/gdp_prefill.h``); this package holds its build step and a thin ctypes
binding.
"""
from .binding import (  # noqa: F401
    GDP_ABI_VERSION,
    GDP_DTYPE_BF16,
    GDP_DTYPE_DEFAULT,
    GDP_DTYPE_F16,
    GDP_DTYPE_F32,
    GDP_DEV_ERR_CU_SEQLENS,
    GDP_DEV_ERR_DESC,
    GDP_DEV_ERR_SLOT,
    GDP_ERR_ALIAS,
    GDP_ERR_CUDA,
    GDP_ERR_INVALID_ARG,
    GDP_ERR_UNSUPPORTED,
    GDP_ERR_WORKSPACE,
    GDP_OK,
    GdpError,
    GdpPrefillArgs,
    LIB_PATH,
    alloc_workspace,
    chunk_gated_delta_product,
    decode_args,
    gated_delta_product_decode,
    gdp_build_descriptors,
    gdp_decode_step,
    gdp_last_error,
    gdp_nt_pad,
    gdp_ntdp_pad,
    gdp_prefill_varlen,
    gdp_prefill_varlen_profiled,
    gdp_prefill_varlen_static_scratch,
    GDP_STATIC_SCRATCH_BYTES,
    gdp_prefill_workspace_bytes,
    load_library,
    make_args,
)
