"""Pins of the oracle's static FP8 (e4m3) quantiser (no GPU).

  * every finite e4m3 code decodes (from the format definition written out
    here in fp64) and re-encodes to itself;
  * the encoder equals torch's float8_e4m3fn conversion of the clamped
    value for every bf16 and every fp16 pattern divided by several scales
    (the clamp to +-448 is the static quantiser's saturation; torch rounds
    to nearest even and gives NaN only past the top rounding boundary);
  * ties between neighbouring codes go to the even code, in the subnormal
    and the normal range, and saturation / NaN / signed zero behave as
    specified;
  * ln_modulate_fp8 is ln_modulate's output passed through quant_e4m3.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp64ref import value16


def decode_e4m3(code):
    code = np.asarray(code, dtype=np.int64)
    s = np.where(code & 0x80, -1.0, 1.0)
    e = (code >> 3) & 0xF
    m = code & 7
    v = np.where(e == 0, m * 2.0 ** -9, (1 + m / 8.0) * 2.0 ** (e - 7))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


def torch_e4m3(f):
    t = torch.from_numpy(np.clip(np.asarray(f, np.float32), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_every_code_round_trips(oracle_lib):
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = decode_e4m3(codes).astype(np.float32)
    assert np.array_equal(oracle.e4m3(vals), codes)
    assert decode_e4m3(0x7E) == 448.0 and decode_e4m3(0x01) == 2.0 ** -9 and decode_e4m3(0x08) == 2.0 ** -6


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("qscale", [1.0, 0.0625, 0.37, 3.0, 1000.0])
def test_quantiser_matches_torch_on_every_pattern(oracle_lib, dtype, qscale):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = value16(pats, dtype)
    pats = pats[~np.isnan(v)]
    got = oracle.quant_e4m3(pats, qscale, dtype)
    with np.errstate(over="ignore"):   # large patterns over small scales overflow to inf: saturated
        f = (value16(pats, dtype).astype(np.float32) / np.float32(qscale)).astype(np.float32)
    assert np.array_equal(got, torch_e4m3(f))


def test_ties_saturation_nan_and_zero(oracle_lib):
    # midpoints between neighbouring codes tie to the even code
    codes = np.arange(0, 0x7E, dtype=np.int64)
    lo, hi = decode_e4m3(codes), decode_e4m3(codes + 1)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)     # exact in binary32
    exp = np.where(codes % 2 == 0, codes, codes + 1).astype(np.uint8)
    assert np.array_equal(oracle.e4m3(mid), exp)
    assert np.array_equal(oracle.e4m3(-mid), exp | 0x80)
    # just above / below a midpoint
    assert np.array_equal(oracle.e4m3(np.nextafter(mid, np.float32(np.inf))), (codes + 1).astype(np.uint8))
    assert np.array_equal(oracle.e4m3(np.nextafter(mid, np.float32(0))), codes.astype(np.uint8))
    special = np.array([448.0, 464.0, 1e30, np.inf, -np.inf, np.nan, -0.0, 0.0, 2.0 ** -10, 2.0 ** -11],
                       dtype=np.float32)
    assert oracle.e4m3(special).tolist() == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F, 0x80, 0x00, 0x00, 0x00]


def test_exact_ties_after_division(oracle_lib):
    # y = m * q with m the midpoint of two neighbouring codes and q a small
    # odd integer: y / q is exactly m (a tie, to the even code); y * (1/q)
    # rounded is not always m, so this fixes the division
    codes = np.arange(0, 0x7E, dtype=np.int64)
    mids = (decode_e4m3(codes) + decode_e4m3(codes + 1)) / 2
    for q in (3, 5, 7, 11, 13):
        y = mids * q
        ok = (y.astype(np.float32).astype(np.float64) == y)
        yb = y[ok].astype(np.float32)
        bf = (yb.view(np.uint32) & 0xFFFF) == 0          # exact in bf16
        pats = (yb[bf].view(np.uint32) >> 16).astype(np.uint16)
        exp = np.where(codes[ok][bf] % 2 == 0, codes[ok][bf], codes[ok][bf] + 1).astype(np.uint8)
        assert pats.size > 20
        assert np.array_equal(oracle.quant_e4m3(pats, float(q)), exp), q


def test_ln_modulate_fp8_is_the_composition(oracle_lib):
    B, N, D = 2, 7, 516
    x = synth.normal_bits(1, B * N * D, 0, 1).reshape(B, N, D)
    t = synth.normal_bits(2, B * 2 * D, 0, 0.1)
    _, y = oracle.ln_modulate(x, B, N, D, (N * D, D, 1), t, D, 2 * D, t, 0, 2 * D, 1e-6)
    _, q = oracle.ln_modulate_fp8(x, B, N, D, (N * D, D, 1), t, D, 2 * D, t, 0, 2 * D, 1e-6, 0.005)
    assert np.array_equal(q, oracle.quant_e4m3(y, 0.005))
    assert (q == 0x7E).any() or (q == 0xFE).any()   # this scale saturates some outputs
