"""Pins of the oracle's RMSNorm chains and of the general norm + modulate
function's broadcast modes (no GPU).

What each test fixes, independently of the oracle's own code:
  * fp64 RMSNorm: the normalised output (scale = shift = 0) is within one
    storage ulp of x / sqrt(mean(x^2) + eps) on every element, for row
    lengths with and without a tail chunk, rows with a nonzero mean, both
    storage types;
  * exact rows: rows built from a pattern whose squares sum to 4 per 8
    elements (eps 0) or 3.75 per 8 (eps 0.25) give rstd = 1/2 exactly, so
    the output is x / 2 exactly; this fixes the divisor D, the eps term and
    the absence of a mean;
  * flipping the signs of any elements flips exactly those outputs: the
    statistic depends on x^2 only (a LayerNorm would move its mean);
  * power-of-two scaling of x (eps = 0) leaves every output bit unchanged;
  * the modulate tail of the RMS mode equals its single-rounding fp64
    definition given the normalised values;
  * the LayerNorm mode equals the pinned ln_modulate, and with a gate the
    pinned gate-add followed by the pinned LN+modulate;
  * per-token modulation rows and per-token [B, S, 1] gates give, row by
    row, the same bits as one-row calls with per-sample rows and a
    broadcast gate row;
  * qk RMSNorm: within the rounding bound of fp64 w * x / rms, exact on the
    exact rows with power-of-two weights.
"""
import numpy as np
import pytest

import oracle
import synth
from fp64ref import FORMATS, bits16, round_to16, ulp_diff, value16

DS = [4, 12, 60, 128, 500, 512, 516, 2240, 3072, 4096, 5120]


def _ulp16(v, dtype):
    p, emin, _ = FORMATS[dtype]
    _, ex = np.frexp(np.abs(np.asarray(v, np.float64)))
    return np.ldexp(1.0, np.maximum(ex - 1, emin) - (p - 1))


def rms(x, B, N, D, sc, sh, eps, dtype="bf16", per_token=False, **kw):
    """x (B, N, D) contiguous; sc / sh (B, D) per sample or (B, N, D) per token."""
    sc = np.ascontiguousarray(sc)
    sh = np.ascontiguousarray(sh)
    if per_token:
        return oracle.norm_scale_shift("rms", x, B, N, D, (N * D, D, 1), sc, 0, N * D, D, sh, 0, N * D, D,
                                       eps, dtype, **kw)
    return oracle.norm_scale_shift("rms", x, B, N, D, (N * D, D, 1), sc, 0, D, 0, sh, 0, D, 0, eps, dtype, **kw)


def rms_fp64(xv, eps):
    x = np.asarray(xv, dtype=np.float64)
    ms = (x * x).mean(axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(np.float32(eps)))


def zeros(shape):
    return np.zeros(shape, dtype=np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", DS)
def test_rms_within_one_ulp_of_fp64(oracle_lib, D, dtype):
    rows = 16
    for seed, (mu, sigma) in enumerate([(0.0, 1.0), (0.7, 2.0), (-3.0, 0.5)]):
        x = synth.normal_bits(500 + 7 * seed + D, rows * D, mu, sigma, dtype).reshape(1, rows, D)
        _, out = rms(x, 1, rows, D, zeros((1, D)), zeros((1, D)), 1e-6, dtype)
        ref = bits16(round_to16(rms_fp64(value16(x, dtype).reshape(rows, D), 1e-6), dtype), dtype)
        d = ulp_diff(out, ref, dtype)
        assert d.max() <= 1, (D, dtype, seed, int(d.max()))


def _exact_rows(D, rows, pattern, seed):
    """Rows of length D (a multiple of 8): each block of 8 is a signed,
    shuffled copy of `pattern`."""
    rng = np.random.default_rng(seed)
    out = np.empty((rows, D), dtype=np.float64)
    for r in range(rows):
        for k in range(0, D, 8):
            blk = np.array(pattern, dtype=np.float64)
            rng.shuffle(blk)
            out[r, k:k + 8] = blk * rng.choice([-1.0, 1.0], 8)
    return out


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [8, 64, 512, 2240, 4096, 5120])
@pytest.mark.parametrize("pattern,eps", [((3, 3, 3, 1, 1, 1, 1, 1), 0.0), ((3, 3, 3, 1, 1, 1, 0, 0), 0.25)])
def test_exact_rows_give_half(oracle_lib, D, dtype, pattern, eps):
    # sum of squares 32 (or 30) per 8 elements: ms = 4 (or 3.75), ms + eps = 4,
    # every square and partial sum an integer below 2^24: rstd = 1/2 exactly
    rows = 6
    xv = _exact_rows(D, rows, pattern, D + int(4 * eps))
    x = bits16(xv, dtype).reshape(1, rows, D)
    _, out, mean, rstd = rms(x, 1, rows, D, zeros((1, D)), zeros((1, D)), eps, dtype, return_stats=True)
    assert np.all(rstd == 0.5) and np.all(mean == 0.0)
    assert np.array_equal(out, bits16(xv / 2 + 0.0, dtype))  # + shift 0 turns -0 into +0


@pytest.mark.parametrize("D", [12, 516, 2240, 4096])
def test_sign_flips_flip_only_those_outputs(oracle_lib, D):
    rows = 8
    x = synth.normal_bits(600 + D, rows * D, 1.5, 1.0).reshape(1, rows, D)
    flip = np.random.default_rng(D).random((1, rows, D)) < 0.3
    xf = np.where(flip, x ^ np.uint16(0x8000), x)
    sc = synth.normal_bits(601 + D, D, 0, 0.1).reshape(1, D)
    _, a = rms(x, 1, rows, D, sc, zeros((1, D)), 1e-6)
    _, b = rms(xf, 1, rows, D, sc, zeros((1, D)), 1e-6)
    fl = flip.reshape(rows, D)
    va, vb = value16(a), value16(b)
    assert np.array_equal(np.where(fl, -va, va), vb)


@pytest.mark.parametrize("D", [60, 2240])
def test_power_of_two_scaling_invariance(oracle_lib, D):
    rows = 8
    x = synth.normal_bits(700 + D, rows * D, 0.3, 1.0).reshape(1, rows, D)
    sc = synth.normal_bits(701 + D, D, 0, 0.1).reshape(1, D)
    sh = synth.normal_bits(702 + D, D, 0, 0.1).reshape(1, D)
    _, base = rms(x, 1, rows, D, sc, sh, 0.0)
    for k in (-3, 5):
        xs = bits16(value16(x) * 2.0 ** k).reshape(1, rows, D)
        _, o = rms(xs, 1, rows, D, sc, sh, 0.0)
        assert np.array_equal(o, base), k


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_modulate_tail_matches_definition(oracle_lib, dtype):
    B, N, D = 2, 8, 516
    x = synth.normal_bits(800, B * N * D, 0, 1, dtype).reshape(B, N, D)
    sc = synth.normal_bits(801, B * D, 0, 0.3, dtype).reshape(B, D)
    sh = synth.normal_bits(802, B * D, 0, 0.3, dtype).reshape(B, D)
    _, y = rms(x, B, N, D, zeros((B, D)), zeros((B, D)), 1e-6, dtype)
    _, out = rms(x, B, N, D, sc, sh, 1e-6, dtype)
    yv = value16(y, dtype).reshape(B, N, D)
    op = round_to16(1.0 + value16(sc, dtype)[:, None, :], dtype)
    p = round_to16(yv * op, dtype)
    ref = bits16(round_to16(p + value16(sh, dtype)[:, None, :], dtype), dtype)
    assert np.array_equal(out, ref.reshape(B * N, D))


def test_layer_mode_is_ln_modulate(oracle_lib):
    B, N, D = 2, 9, 2240
    x = synth.normal_bits(900, B * D * N, 0.5, 1).reshape(B, D, N)  # transposed view
    t = synth.normal_bits(901, B * 2 * D, 0, 0.1)
    a = oracle.ln_modulate(x, B, N, D, (D * N, 1, N), t, D, 2 * D, t, 0, 2 * D, 1e-6)[1]
    b = oracle.norm_scale_shift("layer", x, B, N, D, (D * N, 1, N), t, D, 2 * D, 0, t, 0, 2 * D, 0, 1e-6)[1]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("norm", ["layer", "rms"])
def test_gated_mode_is_gate_add_then_norm(oracle_lib, norm):
    B, N, D = 2, 7, 516
    x = synth.normal_bits(910, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(911, B * N * D, 0, 1).reshape(B, N, D)
    g = synth.normal_bits(912, B * 3 * D, 0, 0.2)  # gate, scale, shift rows per sample
    _, r, out = oracle.norm_scale_shift(norm, x, B, N, D, (N * D, D, 1), g, D, 3 * D, 0, g, 2 * D, 3 * D, 0, 1e-5,
                                        gate=(g, 0, 3 * D, 0, 1), y=y)
    _, r_ref = oracle.residual_gate_add(x, g, 0, 3 * D, y, B, N, D)
    assert np.array_equal(r, r_ref)
    _, o_ref = oracle.norm_scale_shift(norm, r_ref, B, N, D, (N * D, D, 1), g, D, 3 * D, 0, g, 2 * D, 3 * D, 0,
                                       1e-5)
    assert np.array_equal(out, o_ref)
    if norm == "layer":
        _, r2, o2 = oracle.residual_gate_ln_modulate(x, g, 0, 3 * D, y, B, N, D, g, D, 3 * D, g, 2 * D, 3 * D, 1e-5)
        assert np.array_equal(r, r2) and np.array_equal(out, o2)


@pytest.mark.parametrize("norm", ["layer", "rms"])
def test_per_token_rows_and_gates_equal_one_row_calls(oracle_lib, norm):
    # a [B, S, 6D] table: chunk k of token (b, n) at ((b*S + n)*6 + k)*D;
    # gate a per-token scalar [B, S, 1]
    B, N, D = 2, 5, 132
    x = synth.normal_bits(920, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(921, B * N * D, 0, 1).reshape(B, N, D)
    tab = synth.normal_bits(922, B * N * 6 * D, 0, 0.2)
    gs = synth.normal_bits(923, B * N, 0, 0.5)
    _, r, out = oracle.norm_scale_shift(norm, x, B, N, D, (N * D, D, 1), tab, 1 * D, N * 6 * D, 6 * D,
                                        tab, 0, N * 6 * D, 6 * D, 1e-6, gate=(gs, 0, N, 1, 0), y=y)
    for b in range(B):
        for n in range(N):
            row = b * N + n
            t0 = (b * N + n) * 6 * D
            grow = np.full(D, gs[row], dtype=np.uint16)
            _, r1 = oracle.residual_gate_add(x[b, n], grow, 0, 0, y[b, n], 1, 1, D)
            assert np.array_equal(r[row], r1[0])
            _, o1 = oracle.norm_scale_shift(norm, r1, 1, 1, D, (D, D, 1), tab, t0 + D, 0, 0, tab, t0, 0, 0, 1e-6)
            assert np.array_equal(out[row], o1[0]), (b, n)


def test_rms_tail_lanes_add_nothing(oracle_lib):
    # D = 2240: lanes 48..127 own one chunk fewer; zero-padding the row to
    # 2560 changes neither the sum of squares nor, with D fixed, anything else
    row = synth.normal_bits(930, 2240, 0, 1)
    v = value16(row).astype(np.float32)
    ss = oracle.row_sumsq(v, 128)
    pad = np.concatenate([v, np.zeros(320, np.float32)])
    assert ss == oracle.row_sumsq(pad, 128)
    assert abs(ss - float(np.sum(v.astype(np.float64) ** 2))) <= 1e-5 * ss


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("Dh", [64, 100, 128])
def test_qk_rms_within_rounding_bound(oracle_lib, Dh, dtype):
    rows = 200
    x = synth.normal_bits(940 + Dh, rows * Dh, 0.2, 2.0, dtype).reshape(rows, Dh)
    w = synth.normal_bits(941 + Dh, Dh, 1.0, 0.3, dtype)
    _, out = oracle.qk_rmsnorm(x, Dh, w, 1e-6, dtype)
    exact = rms_fp64(value16(x, dtype), 1e-6) * value16(w, dtype)
    err = np.abs(value16(out, dtype) - exact)
    # one storage rounding plus the binary32 statistic and two products
    assert np.all(err <= 0.5 * _ulp16(exact, dtype) + 2e-6 * np.abs(exact) + 1e-30)
    _, plain = oracle.qk_rmsnorm(x, Dh, bits16(np.ones(Dh), dtype), 1e-6, dtype)
    ref = bits16(round_to16(rms_fp64(value16(x, dtype), 1e-6), dtype), dtype)
    assert ulp_diff(plain, ref, dtype).max() <= 1


@pytest.mark.parametrize("Dh", [64, 128])
def test_qk_rms_exact_rows(oracle_lib, Dh):
    rows = 5
    xv = _exact_rows(Dh, rows, (3, 3, 3, 1, 1, 1, 1, 1), Dh)
    wv = 2.0 ** np.random.default_rng(Dh).integers(-2, 3, Dh)
    _, out = oracle.qk_rmsnorm(bits16(xv), Dh, bits16(wv), 0.0)
    assert np.array_equal(out, bits16(xv / 2 * wv))
