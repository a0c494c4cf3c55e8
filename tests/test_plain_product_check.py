"""The static FP8 output takes the code of the product RN(y p) instead of
RN(y / s) when a check over the storage type's significands says the two
agree for every 16-bit value (csrc/quant_e4m3.cuh, quant_plain_share).  The
check compares, for each significand M, the codes of RN(M p) 2^j and
RN(M / s) 2^j at one binade of each rounding class of the e4m3 grid
([2^-11, 2^-10) .. [2^-7, 2^-6), one normal binade, [2^8, 2^9)).  This test
restates that check in numpy and holds it against brute force over all
65536 patterns (oracle encoder, binary32 numpy arithmetic): whenever the
check passes, every code agrees.  For bf16, whose values reach every binade
class at these scales, the converse holds too (the check is not needlessly
strict); fp16 values (2^-24 .. 65504) leave some classes unreached at tiny
scales, where the check may refuse a multiplier that would have served (the
kernel then takes the exact correction).  Candidates are p = RN(1/s) and its
neighbours up to 2 ulp away, as the kernel tries them."""
import numpy as np
import pytest

import oracle
from fp64ref import value16

BINADES = (-11, -10, -9, -8, -7, 0, 8)


def e4(v):
    return oracle.e4m3(np.asarray(v, dtype=np.float32))


def check(s, p, frac_bits):
    M = (1 + np.arange(1 << frac_bits, dtype=np.float64) / (1 << frac_bits)).astype(np.float32)
    qe = (M / np.float32(s)).astype(np.float32)
    q0 = (M * np.float32(p)).astype(np.float32)
    e = np.floor(np.log2(qe.astype(np.float64))).astype(np.int64)
    for b in BINADES:
        a = np.ldexp(qe, b - e).astype(np.float32)
        c = np.ldexp(q0, b - e).astype(np.float32)
        if not np.array_equal(e4(a), e4(c)):
            return False
    return True


def candidates(s):
    r = np.float32(1) / np.float32(s)
    out = []
    for t in range(5):
        k = ((t + 1) >> 1) * (-1 if t & 1 else 1)
        out.append((np.array([r]).view(np.int32) + k).view(np.float32)[0])
    return out


def _scales():
    rng = np.random.default_rng(2024)
    s = list((2.0 ** rng.uniform(-20, 20, 24)).astype(np.float32))
    s += [np.float32(v) for v in (0.03, 0.02, 0.05, 3.0, 5.0, 7.0, 13.0, 0.1, 0.375, 1000.0)]
    return s


@pytest.mark.parametrize("dtype,frac_bits", [("bf16", 7), ("fp16", 10)])
def test_check_matches_brute_force(dtype, frac_bits):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    y = value16(pats, dtype).astype(np.float32)
    y = y[np.isfinite(y)]
    passed = agreed = 0
    for s in _scales():
        if dtype == "fp16" and s > 63.97:
            continue  # the fp16 kernel takes another form there
        for p in candidates(s):
            with np.errstate(all="ignore"):
                truth = np.array_equal(e4((y * p).astype(np.float32)), e4((y / np.float32(s)).astype(np.float32)))
            ok = check(s, p, frac_bits)
            assert truth or not ok, (float(s), float(p))          # sound
            if dtype == "bf16":
                assert ok == truth, (float(s), float(p))          # and exact
            passed += ok
            agreed += truth
    # both outcomes occur over these scales
    assert 0 < passed < len(_scales()) * 5


def test_tie_scales_defeat_every_candidate():
    # y = m s with m an e4m3 midpoint: the product lands on the other side
    # of the tie for some m whatever the multiplier
    for s in (7.0, 13.0):
        assert not any(check(s, p, 7) for p in candidates(s))
    # and 0.03 takes RN(1/s) - 1 ulp
    c = candidates(0.03)
    assert not check(0.03, c[0], 7) and check(0.03, c[1], 7)
