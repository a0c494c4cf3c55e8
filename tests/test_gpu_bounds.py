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


@pytest.mark.parametrize("norm", ["layer", "rms"])
@pytest.mark.parametrize("D,gate", [(516, "scalar"), (4096, "token"), (5120, "sample"), (6140, "scalar"),
                                    (8192, "token"), (3072, None)])
def test_norm_scale_shift_stays_in_bounds(ad, norm, D, gate):
    # per-token rows of a (B, N, 6, D) table; rows kernel up to 6144, general kernel past it
    B, N = 2, 13
    x = synth.normal_bits(D + 1, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(D + 2, B * N * D, 0, 1).reshape(B, N, D)
    tab = synth.normal_bits(D + 3, B * N * 6 * D, 0, 0.2)
    t = dev_tensor(tab).view(B, N, 6, D)
    bo, out = guarded((B, N, D))
    kw, og = {}, None
    if gate is not None:
        br, r = guarded((B, N, D))
        if gate == "scalar":
            gs = synth.normal_bits(D + 4, B * N, 0, 0.5)
            kw = dict(gate=dev_tensor(gs).view(B, N, 1), y=dev_tensor(y), r_out=r)
            og = (gs, 0, N, 1, 0)
        elif gate == "token":
            kw = dict(gate=t[:, :, 2], y=dev_tensor(y), r_out=r)
            og = (tab, 2 * D, N * 6 * D, 6 * D, 1)
        else:
            gr = synth.normal_bits(D + 5, B * D, 0, 0.5)
            kw = dict(gate=dev_tensor(gr).view(B, 1, D), y=dev_tensor(y), r_out=r)
            og = (gr, 0, D, 0, 1)
    ad.norm_scale_shift(dev_tensor(x), t[:, :, 1], t[:, :, 0], 1e-6, norm=norm, out=out, **kw)
    check_guards(bo)
    ref = oracle.norm_scale_shift(norm, x, B, N, D, (N * D, D, 1), tab, D, N * 6 * D, 6 * D, tab, 0, N * 6 * D,
                                  6 * D, 1e-6, gate=og, y=y if gate is not None else None, threads=THREADS)
    if gate is not None:
        check_guards(br)
        assert_bits_equal(host_bits(r).reshape(B * N, D), ref[1], what="r")
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref[-1], what=f"{norm} D={D} gate={gate}")


@pytest.mark.parametrize("rows,Dh", [(1001, 128), (97, 100)])
def test_qk_rmsnorm_stays_in_bounds(ad, rows, Dh):
    q = synth.normal_bits(Dh + 1, rows * Dh, 0, 2).reshape(rows, Dh)
    k = synth.normal_bits(Dh + 2, rows * Dh, 0, 2).reshape(rows, Dh)
    wq, wk = synth.normal_bits(Dh + 3, Dh, 1, 0.05), synth.normal_bits(Dh + 4, Dh, 1, 0.05)
    bq, qo = guarded((rows, Dh))
    bk, ko = guarded((rows, Dh))
    ad.qk_rmsnorm(dev_tensor(q), dev_tensor(k), dev_tensor(wq), dev_tensor(wk), 1e-6, q_out=qo, k_out=ko)
    check_guards(bq)
    check_guards(bk)
    assert_bits_equal(host_bits(qo), oracle.qk_rmsnorm(q, Dh, wq, 1e-6)[1], what="q")
    assert_bits_equal(host_bits(ko), oracle.qk_rmsnorm(k, Dh, wk, 1e-6)[1], what="k")


@pytest.mark.parametrize("D", [3, 1536])
def test_temb_slices_stay_in_bounds(ad, D):
    B, S, K = 2, 11, 6
    table = synth.normal_bits(D + 1, K * D, 0, 0.05)
    temb = synth.normal_bits(D + 2, B * S * K * D, 0, 1)
    n = K * B * S * D
    buf = torch.full((2 * GUARD + n,), float("nan"), dtype=torch.float32, device="cuda")
    canary = buf[:GUARD].clone()
    out = buf[GUARD:GUARD + n].view(K, B, S, D)
    ad.temb_table_slices(dev_tensor(table).view(K, D), dev_tensor(temb).view(B, S, K, D), out=out)
    torch.cuda.synchronize()
    h = buf.cpu().numpy().view(np.uint32)
    cb = canary.cpu().numpy().view(np.uint32)
    assert np.array_equal(h[:GUARD], cb) and np.array_equal(h[-GUARD:], cb)
    ref = oracle.temb_table_slices(table, "bf16", temb, "bf16", B, S, K, D)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("D", [516, 3072, 5120, 8192])
def test_ln_modulate_fp8_stays_in_bounds(ad, D):
    B, N = 2, 9
    x = synth.normal_bits(D + 6, B * N * D, 0, 1).reshape(B, N, D)
    tab = synth.normal_bits(D + 7, B * 2 * D, 0, 0.1).reshape(B, 2, D)
    t = dev_tensor(tab)
    n = B * N * D
    buf = torch.full((2 * 4096 + n,), 0x5A, dtype=torch.uint8, device="cuda")
    out = buf[4096:4096 + n].view(B, N, D)
    qs = torch.tensor([0.02], dtype=torch.float32, device="cuda")
    ad.ln_modulate_fp8(dev_tensor(x), t[:, 1:2], t[:, 0:1], 1e-6, qs, out=out)
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert (h[:4096] == 0x5A).all() and (h[-4096:] == 0x5A).all()
    _, ref = oracle.ln_modulate_fp8(x, B, N, D, (N * D, D, 1), tab, D, 2 * D, tab, 0, 2 * D, 1e-6, 0.02)
    assert np.array_equal(out.cpu().numpy().reshape(B * N, D), ref)
