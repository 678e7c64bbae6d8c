"""Planted mistakes: each mutant of the oracle must fail at least one pin.

Every mutant is a copy of ``oracle/gdp_oracle.c`` with one plausible mistake
written into it (a dropped term, a sign, a row index, the decay placement, a
transposed state, a chunk-state row taken at the wrong time, a descriptor
count), compiled on the CPU into a temporary directory and swapped in for the
real oracle while the pin tests of ``test_oracle_pins`` run.
"""
import ctypes
import inspect
import os
import subprocess

import pytest

import oracle.oracle as orc
from tests import test_oracle_pins as pins

SRC = open(os.path.join(os.path.dirname(orc.__file__), "gdp_oracle.c")).read()

ALPHA = "          const double alpha = !g ? 1.0 : g_is_alpha ? (double)g[t * H + h] : exp((double)g[t * H + h]);\n"
DECAY = ALPHA + "          for (int x = 0; x < nv * K; ++x) S[x] *= alpha;\n"
QLOAD = "load_row(q, t, Hq, h / (H / Hq), K, qkv_f16, use_qk_l2norm, qt);"
ROW = "            const int64_t row = t * M + j;\n"
READOUT = "          /* readout after the last update */\n"

MUTANTS = {
    "sign_of_error": [("b * (vv - pred)", "b * (pred - vv)")],
    "beta_dropped": [("const double b = beta ? (double)beta[row * H + h] : 1.0;", "const double b = 1.0;")],
    "copies_reversed": [(ROW, "            const int64_t row = t * M + (M - 1 - j);\n")],
    "decay_per_subrow": [(ROW, ROW + "            if (j > 0) for (int x = 0; x < nv * K; ++x) S[x] *= alpha;\n")],
    "decay_after_updates": [(DECAY, ALPHA),
                            (READOUT, "          for (int x = 0; x < nv * K; ++x) S[x] *= alpha;\n" + READOUT)],
    "decay_base2": [("exp((double)g[t * H + h])", "exp2((double)g[t * H + h])")],
    "scale_dropped": [("= scale * acc;", "= acc;")],
    "state_transposed": [("(double)src[(int64_t)(v0 + r) * K + d]", "(double)src[(int64_t)d * K + v0 + r]")],
    "q_not_normalised": [(QLOAD, QLOAD.replace("use_qk_l2norm", "0"))],
    "readout_before_updates": [(READOUT, ""),
                               ("          /* n beta-gated Householder updates on the expanded rows t*M + j */\n",
                                READOUT.replace("after the last update", "moved") + "          if (o) {\n"
                                "            " + QLOAD + "\n"
                                "            for (int r = 0; r < nv; ++r) {\n"
                                "              const double *Sr = S + r * K;\n"
                                "              double acc = 0.0;\n"
                                "              for (int d = 0; d < K; ++d) acc += Sr[d] * qt[d];\n"
                                "              o[(t * H + h) * (int64_t)V + v0 + r] = scale * acc;\n"
                                "            }\n          }\n          if (0)\n")],
    "chunk_state_after_decay": [
        ("          if (chunk_states && lt % ORACLE_CHUNK == 0) {", "          if (0) {"),
        ("          /* n beta-gated Householder updates on the expanded rows t*M + j */\n",
         "          if (chunk_states && lt % ORACLE_CHUNK == 0) {\n"
         "            double *dst = chunk_states + (((int64_t)chunk_offsets[i] + lt / ORACLE_CHUNK) * H + h) * KV;\n"
         "            for (int r = 0; r < nv; ++r)\n"
         "              for (int d = 0; d < K; ++d) dst[(int64_t)(v0 + r) * K + d] = S[r * K + d];\n"
         "          }\n")],
    "expanded_count_rescaled": [("ntdp += ceil_div64(L * M, ORACLE_CHUNK);", "ntdp += M * ceil_div64(L, ORACLE_CHUNK);"),
                                ("int64_t n = ceil_div64((cu_seqlens[i + 1] - cu_seqlens[i]) * M, ORACLE_CHUNK);",
                                 "int64_t n = M * ceil_div64(cu_seqlens[i + 1] - cu_seqlens[i], ORACLE_CHUNK);")],
    "cumsum_no_restart": [("if ((r - r0) % ORACLE_CHUNK == 0) acc = 0.0;", "if (r == r0) acc = 0.0;")],
    "cumsum_every_subrow": [("if (g && r % M == 0)", "if (g)")],
    # input variants
    "f16_exponent_bias": [("ldexp((double)(1024 + fr), ex - 25)", "ldexp((double)(1024 + fr), ex - 24)")],
    "f16_subnormals_flushed": [("mag = ldexp((double)fr, -24);", "mag = 0.0;")],
    "f16_flag_ignored": [("return f16 ? widen_f16(bits) : widen_bf16(bits);", "return widen_bf16(bits);")],
    "q_head_modulo": [("load_row(q, t, Hq, h / (H / Hq),", "load_row(q, t, Hq, h % Hq,")],
    "k_head_modulo": [("load_row(k, row, Hk, h / (H / Hk),", "load_row(k, row, Hk, h % Hk,")],
    "v_head_modulo": [("v[(row * Hv + h / (H / Hv))", "v[(row * Hv + h % Hv)")],
    "alpha_exponentiated": [("g_is_alpha ? (double)g[t * H + h]", "g_is_alpha ? exp((double)g[t * H + h])")],
}


def _pin_functions():
    out = []
    for name, fn in inspect.getmembers(pins, inspect.isfunction):
        if not name.startswith("test_"):
            continue
        marks = getattr(fn, "pytestmark", [])
        params = [m for m in marks if m.name == "parametrize"]
        if not params:
            out.append((name, fn, {}))
            continue
        argname, values = params[0].args[0], params[0].args[1]
        for val in values:
            out.append((f"{name}[{val}]", fn, {argname: val}))
    return out


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_mutant_is_caught(mutant, tmp_path):
    src = SRC
    for old, new in MUTANTS[mutant]:
        assert src.count(old) >= 1, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(src)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    real = orc._load()
    lib = ctypes.CDLL(str(so))
    for fname in ("gdp_oracle_forward", "gdp_oracle_descriptors", "gdp_oracle_decay_cumsum", "gdp_oracle_widen_f16"):
        getattr(lib, fname).argtypes = getattr(real, fname).argtypes
        getattr(lib, fname).restype = getattr(real, fname).restype
    caught = []
    saved = orc._lib
    orc._lib = lib
    try:
        for name, fn, kwargs in _pin_functions():
            try:
                if "tmp_path" in inspect.signature(fn).parameters:
                    kwargs = dict(kwargs, tmp_path=tmp_path)
                fn(**kwargs)
            except (AssertionError, ValueError):
                caught.append(name)
            if caught:
                break
    finally:
        orc._lib = saved
    assert caught, f"no pin caught the planted mistake {mutant}"
