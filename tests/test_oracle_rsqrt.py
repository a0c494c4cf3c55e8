"""Pin of the oracle's correctly rounded 1/sqrt against a 100-bit evaluation
(mpmath) rounded once to binary32, plus its scaling law."""
import numpy as np
import pytest

import oracle


def _cr_rsqrt_mp(xs):
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    out = np.empty(len(xs), dtype=np.float32)
    for i, x in enumerate(xs):
        with mpmath.workprec(120):
            y = 1 / mpmath.sqrt(mpmath.mpf(float(x)))
        with mpmath.workprec(24):          # binary32 significand, round to nearest
            y24 = +y                         # results are all in the normal range
        out[i] = np.float32(float(y24))
        _ = mp
    return out


def test_rsqrt_matches_100bit_reference(oracle_lib):
    rng = np.random.default_rng(123)
    bits = rng.integers(1, 0x7F800000, size=6000, dtype=np.uint32)
    special = np.array([1, 2, 3, 0x007FFFFF, 0x00800000, 0x00800001, 0x3F800000, 0x3F800001,
                        0x3F7FFFFF, 0x40000000, 0x40800000, 0x7F7FFFFF, 0x33D6BF95, 0x358637BD],
                       dtype=np.uint32)
    x = np.concatenate([bits, special]).view(np.float32)
    got = oracle.rsqrt_cr(x)
    ref = _cr_rsqrt_mp(x)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_rsqrt_scales_exactly_by_four(oracle_lib):
    rng = np.random.default_rng(7)
    x = rng.uniform(1.0, 4.0, 20000).astype(np.float32)
    a = oracle.rsqrt_cr(x)
    b = oracle.rsqrt_cr(x * np.float32(4.0 ** 10))
    assert np.array_equal(a, b * np.float32(2.0 ** 10))


def test_rsqrt_special_values(oracle_lib):
    x = np.array([0.0, -0.0, np.inf, -1.0, np.nan], dtype=np.float32)
    r = oracle.rsqrt_cr(x)
    assert r[0] == np.inf and r[1] == -np.inf and r[2] == 0.0
    assert np.isnan(r[3]) and np.isnan(r[4])
