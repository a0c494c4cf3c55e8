"""The static FP8 quantisers divide by the scale through div_by_recip
(Markstein's correction from RN(1/b)) instead of CUDA's __fdiv_rn.  This test
runs both on the device for every finite bf16 and fp16 value (the only
numerators the quantisers see) over 44 scales spanning 2^-20 .. 2^20,
including significands of all ones, and checks that the quotients are
bit-identical (hence so are the e4m3 codes), and that numpy's IEEE
division agrees.  It also runs the rows kernel's 4-wide quantiser on every
16-bit pattern against the oracle's codes."""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import oracle
from fp64ref import value16

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("div") / "div_sweep.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-fmad=false", "-shared", os.path.join(HERE, "cuda", "div_sweep.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.div_sweep.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong]
    lib.quant4_sweep.argtypes = [ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return lib


def _scales():
    rng = np.random.default_rng(7)
    s = [1.0, 3.0, 7.0, 0.37, 0.03, 0.004, 1e-6, 2.0 ** -20, 2.0 ** 20, 1000.0]
    s += list((rng.random(24) * 2.0 ** rng.integers(-20, 20, 24)).astype(np.float32))
    ones = np.float32(np.nextafter(np.float32(2.0), np.float32(0)))   # 1.111...1 (binary)
    s += [float(ones * np.float32(2.0 ** k)) for k in (-12, -5, -1, 0, 3, 9, 15)]
    s += [float(np.nextafter(np.float32(1.0), np.float32(2))), 0.1, 0.7]
    return [float(np.float32(v)) for v in s]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_quotients_match_ieee_division(helper, dtype):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    a = value16(pats, dtype).astype(np.float32)
    a = a[np.isfinite(a)]
    ag = torch.from_numpy(a).cuda()
    mine, ieee = torch.empty_like(ag), torch.empty_like(ag)
    for b in _scales():
        assert helper.div_sweep(ag.data_ptr(), b, mine.data_ptr(), ieee.data_ptr(), ag.numel()) == 0
        m, e = mine.cpu().numpy(), ieee.cpu().numpy()
        assert np.array_equal(m.view(np.uint32), e.view(np.uint32)), b
        assert np.array_equal(oracle.e4m3(m), oracle.e4m3(e)), b
        with np.errstate(over="ignore", under="ignore"):
            ref = (a / np.float32(b)).astype(np.float32)         # numpy's IEEE division agrees
        assert np.array_equal(ref.view(np.uint32), e.view(np.uint32)), b


def _tie_scales():
    # scales that put many y / s exactly on e4m3 midpoints (y = m * s exact)
    return [3.0, 5.0, 7.0, 11.0, 13.0, 0.375, 0.625]


def _extreme_scales():
    # outside the branch-free form's range (2^-60 .. 2^60, positive) or, for
    # fp16, above 63.97 (65504 / 1024): the window form only
    return [2.0 ** -70, 2.0 ** 70, -0.03, -3.0, 100.0, 3.0e4]


@pytest.mark.parametrize("form,memo", [(0, 0), (0, 1), (1, 0), (2, 0)],
                         ids=["as_picked", "as_picked_with_memo", "window_form", "corrected_form"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_quantiser_codes_equal_the_oracle(helper, dtype, form, memo):
    """The rows kernel's 4-wide quantisers against the oracle's IEEE division
    and e4m3 encoder, for every 16-bit pattern (NaN codes compared as NaN):
    the form the kernel picks for each scale (the plain product RN(y r) when
    the per-CTA check over all significands passes; else, for an ordinary
    positive scale, clamped magnitudes and Markstein's correction on -y; else
    the window form: the product and the exact quotient near e4m3
    boundaries), and the window and corrected forms forced.  With the memo
    each scale runs twice: the first call searches (the previous scale is
    another), the second takes the memo's outcome."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    yg = torch.from_numpy(pats.view(np.int16).copy()).cuda()
    codes = torch.empty(65536, dtype=torch.uint8, device="cuda")
    picked = torch.zeros(1, dtype=torch.int32, device="cuda")
    plain_for = {}
    scales = _scales() + _tie_scales() + _extreme_scales()
    for s in [v for v in scales for _ in range(1 + memo)]:
        assert helper.quant4_sweep(yg.data_ptr(), s, codes.data_ptr(), 65536 // 4, int(dtype == "fp16"), form, memo,
                                   picked.data_ptr()) == 0
        expect_fast = 2.0 ** -60 <= s <= 2.0 ** 60 and (dtype == "bf16" or s <= 65504.0 / 1024.0)
        pk = int(picked.item())
        assert bool(pk & 1) == expect_fast, s
        assert not (pk & 2) or expect_fast, s
        assert plain_for.get(s, bool(pk & 2)) == bool(pk & 2), s   # the memo's outcome is the search's
        plain_for[s] = bool(pk & 2)
        if form == 2 and not expect_fast:
            continue  # the corrected form is defined for ordinary positive scales only
        got = codes.cpu().numpy()
        ref = oracle.quant_e4m3(pats, s, dtype)
        nan_r = (ref & 0x7F) == 0x7F
        assert np.array_equal((got & 0x7F) == 0x7F, nan_r), s
        assert np.array_equal(got[~nan_r], ref[~nan_r]), (s, int((got[~nan_r] != ref[~nan_r]).sum()))
    # exact ties that the product rounds the other way (y = m s, s = 7, 13)
    # defeat every multiplier tried; 0.03 takes r - 1 ulp; nearly every other
    # ordinary scale takes the product
    assert not plain_for[7.0] and not plain_for[13.0]
    assert plain_for[float(np.float32(0.03))]
    fast_scales = [s for s in _scales() if 2.0 ** -60 <= s <= 2.0 ** 60 and (dtype == "bf16" or s <= 63.97)]
    assert sum(plain_for[s] for s in fast_scales) >= 0.9 * len(fast_scales)
