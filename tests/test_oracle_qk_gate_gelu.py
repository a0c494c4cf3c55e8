"""Pins of the oracle's qk_head_layernorm, residual_gate_add and
bias_gelu_tanh (no GPU).

  qk_head_layernorm: the normalised value before the affine is within one
      ulp of an fp64 two-pass LayerNorm; the affine output is within the
      single rounding of fma(w, u, b) plus the propagated ulp of u; w = 1,
      b = 0 reduces to plain LN; rows shorter than 128 (masked lanes) too.
  residual_gate_add: the two-step rounding equals the single-rounding fp64
      definition on 100 % of elements (the double rounding through binary32
      is innocuous for one bf16/fp16 product or sum), and gate = 0 returns x.
  bias_gelu_tanh: the 65536-entry table of each dtype equals a 120-bit
      evaluation of 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))) rounded
      to binary32 and then to storage; G(0) = 0, G(v) = v for large v,
      G(+inf) = +inf, G(-inf) and G(NaN) are NaN; the bias add rounds once.
"""
import numpy as np
import pytest

import oracle
import synth
from fp64ref import FORMATS, bits16, ln_fp64, round_to16, ulp_diff, value16


# ----------------------------------------------------------------- qk LN

@pytest.mark.parametrize("Dh", [4, 32, 64, 100, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_qk_plain_ln_within_one_ulp(oracle_lib, Dh, dtype):
    rows = 512
    x = synth.normal_bits(7 + Dh, rows * Dh, 0, 2, dtype).reshape(rows, Dh)
    one = bits16(np.ones(Dh), dtype)
    zero = np.zeros(Dh, np.uint16)
    _, out = oracle.qk_head_layernorm(x, Dh, one, zero, 1e-6, dtype)
    y64, _, _ = ln_fp64(value16(x, dtype), 1e-6)
    d = ulp_diff(out, bits16(round_to16(y64, dtype), dtype), dtype)
    assert d.max() <= 1


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_qk_affine_within_rounding_bound(oracle_lib, dtype):
    rows, Dh = 1024, 128
    x = synth.normal_bits(17, rows * Dh, 0, 2, dtype).reshape(rows, Dh)
    w = synth.normal_bits(18, Dh, 1, 0.05, dtype)
    b = synth.normal_bits(19, Dh, 0, 0.05, dtype)
    _, out = oracle.qk_head_layernorm(x, Dh, w, b, 1e-6, dtype)
    u64, _, _ = ln_fp64(value16(x, dtype), 1e-6)
    exact = value16(w, dtype) * u64 + value16(b, dtype)
    got = value16(out, dtype)
    p, emin, _ = FORMATS[dtype]
    _, ex = np.frexp(np.abs(exact))
    ulp = np.ldexp(1.0, np.maximum(ex - 1, emin) - (p - 1))
    # one storage rounding of the result plus the binary32 error of u (a few
    # ulps of 2^-24 relative) scaled by |w|
    bound = ulp + np.abs(value16(w, dtype)) * np.abs(u64) * 2.0 ** -20
    assert np.all(np.abs(got - exact) <= bound)
    d = ulp_diff(out, bits16(round_to16(exact, dtype), dtype), dtype)
    assert (d == 0).mean() > 0.999


def test_qk_rows_are_independent(oracle_lib):
    rows, Dh = 300, 128
    x = synth.normal_bits(27, rows * Dh, 0, 2).reshape(rows, Dh)
    w = synth.normal_bits(28, Dh, 1, 0.05)
    b = synth.normal_bits(29, Dh, 0, 0.05)
    _, full = oracle.qk_head_layernorm(x, Dh, w, b, 1e-6)
    ids, part = oracle.qk_head_layernorm(x, Dh, w, b, 1e-6, rows=[299, 0, 150], threads=2)
    assert np.array_equal(part, full[ids])
    _, thr = oracle.qk_head_layernorm(x, Dh, w, b, 1e-6, threads=4)
    assert np.array_equal(thr, full)


# ------------------------------------------------------------- gate add

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gate_add_equals_single_rounding_definition(oracle_lib, dtype):
    B, N, D = 2, 64, 4096
    x = synth.normal_bits(37, B * N * D, 0, 1, dtype).reshape(B, N, D)
    y = synth.normal_bits(38, B * N * D, 0, 1, dtype).reshape(B, N, D)
    g = synth.normal_bits(39, B * D, 0, 0.1, dtype).reshape(B, D)
    _, out = oracle.residual_gate_add(x, g, 0, D, y, B, N, D, dtype)
    gy = round_to16(value16(g, dtype)[:, None, :] * value16(y, dtype), dtype)
    ref = bits16(round_to16(value16(x, dtype) + gy, dtype), dtype).reshape(B * N, D)
    assert np.array_equal(value16(out, dtype), value16(ref, dtype))


def test_gate_zero_returns_x(oracle_lib):
    B, N, D = 1, 32, 512
    x = synth.normal_bits(47, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(48, B * N * D, 0, 1).reshape(B, N, D)
    g = np.zeros((B, D), np.uint16)
    _, out = oracle.residual_gate_add(x, g, 0, D, y, B, N, D)
    assert np.array_equal(value16(out), value16(x.reshape(B * N, D)))


# ------------------------------------------------------------------ GELU

def _gelu_reference_table(dtype):
    mpmath = pytest.importorskip("mpmath")
    h = np.arange(1 << 16, dtype=np.uint16)
    v = value16(h, dtype)
    out32 = np.empty(v.size, dtype=np.float32)
    k0 = None
    with mpmath.workprec(200):
        k0 = mpmath.sqrt(2 / mpmath.pi)
        k1 = mpmath.mpf(44715) / 1000000
    for i, vi in enumerate(v):
        if not np.isfinite(vi):
            out32[i] = np.inf if vi == np.inf else np.nan
            continue
        with mpmath.workprec(200):
            m = mpmath.mpf(float(vi))
            z = k0 * (m + k1 * m ** 3)
            g = m / (1 + mpmath.exp(-2 * z))
            a = abs(g)
            if a == 0:
                out32[i] = np.copysign(np.float32(0.0), np.float32(vi))   # G(-0) = -0
                continue
            if a < mpmath.ldexp(1, -126):       # binary32 subnormal: fixed quantum 2^-149
                q = mpmath.nint(mpmath.ldexp(g, 149))
                out32[i] = np.float32(float(mpmath.ldexp(q, -149))) if q != 0 else \
                    np.copysign(np.float32(0.0), np.float32(vi))
                continue
        with mpmath.workprec(24):
            g24 = +g
        out32[i] = np.float32(float(g24)) if abs(float(g24)) < 3.5e38 else np.float32(np.inf)
    ref = np.empty(v.size, dtype=np.uint16)
    nan = np.isnan(out32)
    ref[~nan] = bits16(round_to16(out32[~nan].astype(np.float64), dtype), dtype)
    ref[nan] = 0x7FC0 if dtype == "bf16" else 0x7E00
    return ref


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gelu_table_matches_high_precision(oracle_lib, dtype):
    table = oracle.gelu_table(dtype)
    ref = _gelu_reference_table(dtype)
    assert np.array_equal(table, ref)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gelu_special_points(oracle_lib, dtype):
    t = oracle.gelu_table(dtype)
    inf = 0x7F80 if dtype == "bf16" else 0x7C00
    nan_pat = 0x7FC0 if dtype == "bf16" else 0x7E00
    assert t[0] == 0 and t[inf] == inf
    assert t[inf | 0x8000] == nan_pat and t[nan_pat] == nan_pat
    big = bits16(np.array([20.0, 100.0, 1000.0]), dtype)
    assert np.array_equal(t[big], big)
    neg = value16(t[bits16(np.array([-20.0, -100.0]), dtype)], dtype)
    assert np.all(neg == 0) and np.all(np.signbit(neg))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_bias_gelu_rounds_the_sum_once(oracle_lib, dtype):
    rows, width = 64, 1000
    x = synth.normal_bits(57, rows * width, 0, 1, dtype).reshape(rows, width)
    bias = synth.normal_bits(58, width, 0, 0.02, dtype)
    _, out = oracle.bias_gelu_tanh(x, bias, rows, width, dtype)
    v = bits16(round_to16(value16(x, dtype) + value16(bias, dtype), dtype), dtype)
    assert np.array_equal(out, oracle.gelu_table(dtype)[v])
    ids, part = oracle.bias_gelu_tanh(x, bias, rows, width, dtype, rows=[63, 5], threads=2)
    assert np.array_equal(part, out[ids])
