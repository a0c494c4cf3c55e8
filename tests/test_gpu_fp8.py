"""GPU parity of adaln_ln_modulate_fp8 (LayerNorm + adaLN modulate into
static FP8 e4m3) with the oracle, through the C ABI: every code equal, NaN
codes compared as NaN (sign and payload unspecified), on the rows kernel
and the general kernel, with scales that keep every value in range and
scales that saturate."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import THREADS, dev_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ad():
    import adaln_modulate_gb300
    assert torch.cuda.is_available()
    return adaln_modulate_gb300


def assert_codes_equal(got, ref, what=""):
    got = np.asarray(got, np.uint8).reshape(-1)
    ref = np.asarray(ref, np.uint8).reshape(-1)
    nan_g, nan_r = (got & 0x7F) == 0x7F, (ref & 0x7F) == 0x7F
    assert np.array_equal(nan_g, nan_r), f"{what}: NaN positions differ"
    bad = (got != ref) & ~nan_r
    assert not bad.any(), f"{what}: {int(bad.sum())} of {got.size} codes differ, first at {np.argmax(bad)}"


def case(ad, B, N, D, qscale, dtype="bf16", seed=0, layout="rows", expect=None, rows=None, x_bits=None,
         tab_bits=None):
    if layout == "tokens":
        xb = synth.normal_bits(seed, B * D * N, 0.2, 1, dtype) if x_bits is None else x_bits
        strides = (D * N, 1, N)
        x = dev_tensor(xb, dtype).view(B, D, N).permute(0, 2, 1)
    else:
        xb = synth.normal_bits(seed, B * N * D, 0.2, 1, dtype) if x_bits is None else x_bits
        strides = (N * D, D, 1)
        x = dev_tensor(xb, dtype).view(B, N, D)
    tab = synth.normal_bits(seed + 1, B * 2 * D, 0, 0.2, dtype) if tab_bits is None else tab_bits
    t = dev_tensor(tab, dtype).view(B, 2, D)
    qs = torch.tensor([qscale], dtype=torch.float32, device="cuda")
    variant = ad.ln_modulate_fp8_variant(x, t[:, 1:2], t[:, 0:1], 1e-6, qs)
    if expect:
        assert variant == expect, variant
    out = ad.ln_modulate_fp8(x, t[:, 1:2], t[:, 0:1], 1e-6, qs)
    torch.cuda.synchronize()
    ids, ref = oracle.ln_modulate_fp8(xb, B, N, D, strides, tab, D, 2 * D, tab, 0, 2 * D, 1e-6, qscale, dtype,
                                      rows=rows, threads=THREADS)
    got = out.view(torch.uint8).cpu().numpy().reshape(B * N, D)[ids]
    assert_codes_equal(got, ref, f"B={B} N={N} D={D} {dtype} s={qscale} {layout} -> {variant}")
    return ref


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [4, 12, 516, 2240, 3072, 4096])
def test_rows_kernel(ad, D, dtype):
    case(ad, 3, 29, D, 0.02, dtype, seed=D, expect="rows")


@pytest.mark.parametrize("qscale", [1.0, 0.37, 0.004, 7.0])
def test_scales_in_range_and_saturating(ad, qscale):
    ref = case(ad, 2, 40, 3072, qscale, seed=int(qscale * 1000) + 3, expect="rows")
    if qscale == 0.004:
        assert ((ref & 0x7F) == 0x7E).any()   # saturated codes present


@pytest.mark.parametrize("dtype,qscale", [("bf16", 0.03), ("bf16", 7.0), ("bf16", -0.05), ("fp16", 0.03),
                                          ("fp16", 13.0), ("fp16", 100.0)])
def test_each_quantiser_form(ad, dtype, qscale):
    # the rows kernel's output pass in each of its forms: the plain product
    # (0.03, with the multiplier RN(1/s) - 1 ulp), the clamped correction
    # (7 and 13: exact ties defeat every multiplier), the window form (a
    # negative scale; fp16 with a scale above 63.97)
    case(ad, 2, 40, 3072, qscale, dtype, seed=int(abs(qscale) * 100) + 5, expect="rows")


@pytest.mark.parametrize("D,expect", [(5120, "rows"), (6144, "rows"), (8192, "generic")])
def test_large_d(ad, D, expect):
    case(ad, 2, 11, D, 0.02, seed=D + 1, expect=expect)


def test_transposed_view_takes_the_general_kernel(ad):
    case(ad, 2, 48, 2240, 0.05, seed=7, layout="tokens", expect="generic")


def test_non_finite_rows(ad):
    B, N, D = 1, 6, 512
    xb = synth.normal_bits(9, B * N * D, 0, 1)
    xb[2 * D + 5] = 0x7F80          # +inf in row 2: that row becomes NaN
    xb[4 * D + 7] = 0x7FC0          # NaN in row 4
    ref = case(ad, B, N, D, 0.05, seed=9, x_bits=xb, expect="rows")
    assert ((ref[2] & 0x7F) == 0x7F).all() and ((ref[4] & 0x7F) == 0x7F).all()


def test_flux_like_shape_sampled_rows(ad):
    case(ad, 1, 4608, 3072, 0.03, seed=11, expect="rows")


@pytest.mark.parametrize("D", [3072, 2240])
@pytest.mark.parametrize("qscale", [1e-30, 1e30])
def test_scales_outside_the_division_window(ad, qscale, D):
    # most quotients leave the range where the reciprocal correction is exact
    # (huge ones saturate, tiny ones round to zero): whole rows take the
    # checked quotient, on full and ragged widths
    case(ad, 2, 40, D, qscale, seed=int(D + (qscale > 1)), expect="rows")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_exact_zero_outputs(ad, dtype):
    # constant rows normalise to 0, so their outputs are 0 * op + shift: the
    # +0 shift columns and the -0 ones with op = -1 give signed-zero outputs
    # (outside the division window) beside ordinary values; random rows in
    # between take the unchecked quotient in the same warps
    B, N, D = 1, 16, 3072
    xb = synth.normal_bits(21, B * N * D, 0.2, 1, dtype).reshape(N, D)
    one = 0x3F80 if dtype == "bf16" else 0x3C00
    xb[0::3] = one
    tab = synth.normal_bits(22, B * 2 * D, 0, 0.2, dtype)
    tab[0:D:5] = 0x0000
    tab[3:D:7] = 0x8000
    tab[D + 3:2 * D:7] = 0xC000   # scale -2: op = -1, so 0 * op = -0 and -0 + -0 = -0
    ref = case(ad, B, N, D, 0.05, dtype, seed=21, x_bits=xb.reshape(-1), tab_bits=tab, expect="rows")
    assert (ref[0] == 0x00).any() and (ref[0] == 0x80).any()
