"""Bounds: every op writes its output into the middle of a larger buffer whose
4 KiB on each side hold a canary pattern; the canaries must be untouched and
the output must still match the oracle.  Shapes with ragged tails, several
tiles per CTA and both kernels of each layout."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import THREADS, assert_bits_equal, dev_tensor, host_bits

pytestmark = pytest.mark.gpu
GUARD = 2048  # elements = 4 KiB of 16-bit values
CANARY = 0x7A5C


@pytest.fixture(scope="module")
def ad():
    import adaln_modulate_gb300
    assert torch.cuda.is_available()
    return adaln_modulate_gb300


def guarded(shape, dtype=torch.bfloat16):
    n = int(np.prod(shape))
    buf = torch.full((GUARD + n + GUARD,), CANARY, dtype=torch.int16, device="cuda").view(dtype)
    return buf, buf[GUARD:GUARD + n].view(shape)


def check_guards(buf):
    torch.cuda.synchronize()
    h = buf.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (h[:GUARD] == CANARY).all(), "write before the output"
    assert (h[-GUARD:] == CANARY).all(), "write after the output"


@pytest.mark.parametrize("B,N,D,layout", [(2, 37, 516, "rows"), (3, 41, 4096, "rows"), (1, 9, 12, "rows"),
                                          (2, 24, 2244, "tokens"), (3, 1000, 1024, "tokens"),
                                          (2, 16, 5632, "tokens"), (2, 5, 516, "generic")])
def test_ln_modulate_stays_in_bounds(ad, B, N, D, layout):
    if layout == "tokens":
        xb = synth.normal_bits(D, B * D * N, 0, 1).reshape(B, D, N)
        strides = (D * N, 1, N)
        xv = dev_tensor(xb).permute(0, 2, 1)
    elif layout == "generic":
        xb = synth.normal_bits(D, 3 * B * N * D, 0, 1)
        strides = (3 * N * D, 3 * D, 3)
        xv = torch.as_strided(dev_tensor(xb), (B, N, D), strides)
    else:
        xb = synth.normal_bits(D, B * N * D, 0, 1).reshape(B, N, D)
        strides = (N * D, D, 1)
        xv = dev_tensor(xb)
    table = synth.normal_bits(D + 1, B * 2 * D, 0, 0.1).reshape(B, 2, D)
    tg = dev_tensor(table)
    buf, out = guarded((B, N, D))
    ad.ln_modulate(xv, tg[:, 1:2], tg[:, 0:1], 1e-6, out=out)
    check_guards(buf)
    _, ref = oracle.ln_modulate(xb, B, N, D, strides, table, D, 2 * D, table, 0, 2 * D, 1e-6, threads=THREADS)
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref, what=f"{layout} D={D}")


@pytest.mark.parametrize("rows,Dh", [(1001, 128), (333, 64), (97, 100)])
def test_qk_stays_in_bounds(ad, rows, Dh):
    q = synth.normal_bits(Dh, rows * Dh, 0, 2).reshape(rows, Dh)
    k = synth.normal_bits(Dh + 8, rows * Dh, 0, 2).reshape(rows, Dh)
    w = [synth.normal_bits(Dh + s, Dh, m, 0.05) for s, m in ((3, 1.0), (4, 0.0), (5, 1.0), (6, 0.0))]
    bq, qo = guarded((rows, Dh))
    bk, ko = guarded((rows, Dh))
    ad.qk_head_layernorm(dev_tensor(q), dev_tensor(k), *[dev_tensor(v) for v in w], 1e-6, q_out=qo, k_out=ko)
    check_guards(bq)
    check_guards(bk)
    assert_bits_equal(host_bits(qo), oracle.qk_head_layernorm(q, Dh, w[0], w[1], 1e-6)[1], what="q")
    assert_bits_equal(host_bits(ko), oracle.qk_head_layernorm(k, Dh, w[2], w[3], 1e-6)[1], what="k")


@pytest.mark.parametrize("D", [3, 100, 4097])
def test_gate_and_gelu_stay_in_bounds(ad, D):
    B, N = 2, 21
    x = synth.normal_bits(D, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(D + 9, B * N * D, 0, 1).reshape(B, N, D)
    g = synth.normal_bits(D + 10, B * D, 0, 0.1).reshape(B, 1, D)
    buf, out = guarded((B, N, D))
    ad.residual_gate_add(dev_tensor(x), dev_tensor(g), dev_tensor(y), out=out)
    check_guards(buf)
    assert_bits_equal(host_bits(out).reshape(B * N, D), oracle.residual_gate_add(x, g, 0, D, y, B, N, D)[1],
                      what="gate")
    bias = synth.normal_bits(D + 7, D, 0, 0.02)
    buf, out = guarded((B * N, D))
    ad.bias_gelu_tanh(dev_tensor(x).view(B * N, D), dev_tensor(bias), out=out)
    check_guards(buf)
    assert_bits_equal(host_bits(out), oracle.bias_gelu_tanh(x, bias, B * N, D)[1], what="gelu")


@pytest.mark.parametrize("D", [516, 4096, 4100])
def test_residual_ln_stays_in_bounds(ad, D):
    B, N = 2, 23
    x = synth.normal_bits(D, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(D + 9, B * N * D, 0, 1).reshape(B, N, D)
    gsc = synth.normal_bits(D + 1, B * 3 * D, 0, 0.1).reshape(B, 3, D)
    tg = dev_tensor(gsc)
    br, r = guarded((B, N, D))
    bo, out = guarded((B, N, D))
    ad.residual_gate_ln_modulate(dev_tensor(x), tg[:, 0:1], dev_tensor(y), tg[:, 1:2], tg[:, 2:3], 1e-5,
                                 r_out=r, out=out)
    check_guards(br)
    check_guards(bo)
    _, r_ref, o_ref = oracle.residual_gate_ln_modulate(x, gsc, 0, 3 * D, y, B, N, D, gsc, D, 3 * D, gsc, 2 * D,
                                                       3 * D, 1e-5, threads=THREADS)
    assert_bits_equal(host_bits(r).reshape(B * N, D), r_ref, what="r")
    assert_bits_equal(host_bits(out).reshape(B * N, D), o_ref, what="out")
