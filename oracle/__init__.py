"""Float64 CPU oracle for the chunked Gated DeltaProduct prefill: forward pass and its backward.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``, never by the product package.  It shares no
code with the CUDA path.  See ``oracle/gdp_oracle.c`` for the definition followed.
"""
from .oracle import (  # noqa: F401
    L2_EPS,
    CHUNK,
    backward,
    build_oracle,
    decay_cumsum,
    descriptors,
    forward,
    oracle_threads,
    widen_f16,
)
