"""GPU parity of the general norm + modulate (LayerNorm or RMSNorm, per-sample
or per-token modulation rows, optional residual gate with per-sample rows,
per-token rows or one value per token) and of the per-head QK RMSNorm with
the oracle, bit for bit, through the C ABI.  Each case also checks which
kernel the call takes, so the fast paths are the ones being compared."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import THREADS, assert_bits_equal, dev_tensor, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ad():
    import adaln_modulate_gb300
    assert torch.cuda.is_available()
    return adaln_modulate_gb300


def case(ad, norm, B, N, D, dtype="bf16", seed=0, per_token=False, gate=None, in_place=None,
         layout="rows", rows=None, eps=1e-6, expect=None):
    """gate: None, "sample" (one row per sample), "token" (one row per token)
    or "scalar" (one value per token).  per_token: scale / shift are chunks of
    a (B, N, 6, D) table; otherwise chunks of a (B, 6, D) table.
    layout "rows" (contiguous x) or "tokens" (the transposed view of a
    contiguous (B, D, N) tensor)."""
    if layout == "tokens":
        xb = synth.normal_bits(seed, B * D * N, 0.3, 1, dtype)
        strides = (D * N, 1, N)
        x = dev_tensor(xb, dtype).view(B, D, N).permute(0, 2, 1)
    else:
        xb = synth.normal_bits(seed, B * N * D, 0.3, 1, dtype)
        strides = (N * D, D, 1)
        x = dev_tensor(xb, dtype).view(B, N, D)
    if per_token:
        tab = synth.normal_bits(seed + 1, B * N * 6 * D, 0, 0.2, dtype)
        t = dev_tensor(tab, dtype).view(B, N, 6, D)
        sc, sh = t[:, :, 1], t[:, :, 0]
        sc_args = (tab, D, N * 6 * D, 6 * D)
        sh_args = (tab, 0, N * 6 * D, 6 * D)
    else:
        tab = synth.normal_bits(seed + 1, B * 6 * D, 0, 0.2, dtype)
        t = dev_tensor(tab, dtype).view(B, 6, D)
        sc, sh = t[:, 1:2], t[:, 0:1]
        sc_args = (tab, D, 6 * D, 0)
        sh_args = (tab, 0, 6 * D, 0)
    kw, og = {}, None
    if gate is not None:
        yb = synth.normal_bits(seed + 2, B * N * D, 0, 1, dtype)
        y = dev_tensor(yb, dtype).view(B, N, D)
        if gate == "scalar":
            gb = synth.normal_bits(seed + 3, B * N, 0, 0.5, dtype)
            g = dev_tensor(gb, dtype).view(B, N, 1)
            og = (gb, 0, N, 1, 0)
        elif gate == "token":
            g = t[:, :, 2] if per_token else None
            if g is None:
                gb = synth.normal_bits(seed + 3, B * N * D, 0, 0.5, dtype)
                g = dev_tensor(gb, dtype).view(B, N, D)
                og = (gb, 0, N * D, D, 1)
            else:
                og = (tab, 2 * D, N * 6 * D, 6 * D, 1)
        else:
            g = t[:, :, 2] if per_token else t[:, 2:3]
            og = (tab, 2 * D, N * 6 * D if per_token else 6 * D, 6 * D if per_token else 0, 1)
        kw = dict(gate=g, y=y, r_out={"x": x, "y": y}.get(in_place))
    variant = ad.norm_scale_shift_variant(x, sc, sh, eps, norm=norm, **kw)
    if expect is not None:
        assert variant == expect, variant
    res = ad.norm_scale_shift(x, sc, sh, eps, norm=norm, **kw)
    torch.cuda.synchronize()
    ref = oracle.norm_scale_shift(norm, xb, B, N, D, strides, *sc_args, *sh_args, eps, dtype, gate=og,
                                  y=yb if gate is not None else None, rows=rows, threads=THREADS)
    what = f"{norm} B={B} N={N} D={D} {dtype} per_token={per_token} gate={gate} {layout} -> {variant}"
    if gate is None:
        ids, o_ref = ref
        assert_bits_equal(host_bits(res).reshape(B * N, D)[ids], o_ref, dtype, what)
    else:
        ids, r_ref, o_ref = ref
        r, out = res
        assert_bits_equal(host_bits(r).reshape(B * N, D)[ids], r_ref, dtype, "r: " + what)
        assert_bits_equal(host_bits(out).reshape(B * N, D)[ids], o_ref, dtype, "out: " + what)
    return variant


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [4, 12, 512, 516, 2240, 3072, 4096])
def test_rms_rows_kernel(ad, D, dtype):
    case(ad, "rms", 3, 37, D, dtype, seed=D, expect="rows")


@pytest.mark.parametrize("D", [4100, 5120, 6144, 8192])
def test_rms_large_d(ad, D):
    case(ad, "rms", 2, 19, D, seed=D + 1, expect="rows" if D <= 6144 else "generic")


def test_rms_transposed_view_takes_the_general_kernel(ad):
    case(ad, "rms", 2, 40, 2240, seed=5, layout="tokens", expect="generic")


@pytest.mark.parametrize("norm", ["layer", "rms"])
@pytest.mark.parametrize("D", [516, 3072, 5120])
def test_per_token_modulation_rows(ad, norm, D):
    case(ad, norm, 2, 33, D, seed=D + 7, per_token=True, expect="rows" if D <= 6144 else "generic")


@pytest.mark.parametrize("norm", ["layer", "rms"])
@pytest.mark.parametrize("gate", ["sample", "token", "scalar"])
@pytest.mark.parametrize("D", [12, 2240, 4096, 5120, 8192])
def test_gated(ad, norm, gate, D):
    case(ad, norm, 2, 21, D, seed=D + 11, gate=gate, per_token=(gate == "token"),
         expect="rows" if D <= 6144 else "generic")


@pytest.mark.parametrize("norm", ["layer", "rms"])
def test_gated_per_sample_modulation_with_per_token_gates(ad, norm):
    # per-sample scale / shift in the shared table, gate per token (row or scalar)
    case(ad, norm, 2, 30, 1024, seed=21, gate="scalar", expect="rows")
    case(ad, norm, 2, 30, 1024, seed=22, gate="token", expect="rows")


@pytest.mark.parametrize("in_place", ["x", "y"])
def test_gated_in_place(ad, in_place):
    case(ad, "rms", 2, 25, 2048, seed=31, gate="scalar", per_token=True, in_place=in_place, expect="rows")
    case(ad, "layer", 2, 25, 5120, seed=32, gate="token", per_token=True, in_place=in_place, expect="rows")
    case(ad, "layer", 2, 25, 8192, seed=33, gate="token", per_token=True, in_place=in_place, expect="generic")


@pytest.mark.parametrize("B,D", [(2, 2728), (2, 2732), (4, 1364), (8, 1024)])
def test_rms_gated_shared_table_edge(ad, B, D):
    case(ad, "rms", B, 9, D, seed=B * D, gate="sample", expect="rows")


def test_rms_fp16_gated_per_token(ad):
    case(ad, "rms", 2, 17, 3072, "fp16", seed=41, gate="scalar", per_token=True, expect="rows")


def test_layer_mode_equals_ln_modulate(ad):
    B, N, D = 2, 64, 2240
    x = dev_tensor(synth.normal_bits(51, B * N * D, 0, 1)).view(B, N, D)
    t = dev_tensor(synth.normal_bits(52, B * 6 * D, 0, 0.1)).view(B, 6, D)
    a = ad.ln_modulate(x, t[:, 1:2], t[:, 0:1], 1e-6)
    b = ad.norm_scale_shift(x, t[:, 1:2], t[:, 0:1], 1e-6, norm="layer")
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(a), host_bits(b))


def test_rmsnorm_scale_shift_entry_point(ad):
    B, N, D = 2, 50, 3072
    xb = synth.normal_bits(61, B * N * D, 0, 1)
    tab = synth.normal_bits(62, B * N * 6 * D, 0, 0.2)
    t = dev_tensor(tab).view(B, N, 6, D)
    out = ad.rmsnorm_scale_shift(dev_tensor(xb).view(B, N, D), t[:, :, 1], t[:, :, 0], 1e-6)
    torch.cuda.synchronize()
    _, ref = oracle.norm_scale_shift("rms", xb, B, N, D, (N * D, D, 1), tab, D, N * 6 * D, 6 * D, tab, 0,
                                     N * 6 * D, 6 * D, 1e-6, threads=THREADS)
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref, what="rmsnorm_scale_shift")


def test_ltx2_like_shape_sampled_rows(ad):
    # 4096-wide rows, 6144 tokens per sample, per-token modulation, sampled rows
    case(ad, "rms", 1, 6144, 4096, seed=71, per_token=True, expect="rows")


def qk_case(ad, rows, Dh, dtype="bf16", seed=0, offset=0, which="both"):
    q = synth.normal_bits(seed, rows * Dh, 0.3, 2, dtype).reshape(rows, Dh)
    k = synth.normal_bits(seed + 1, rows * Dh, -0.2, 1.5, dtype).reshape(rows, Dh)
    wq = synth.normal_bits(seed + 2, Dh, 1.0, 0.1, dtype)
    wk = synth.normal_bits(seed + 3, Dh, 1.0, 0.1, dtype)

    def dev(bits):
        # offset elements into a larger buffer (offset 4: 8-byte but not 16-byte aligned)
        buf = dev_tensor(np.concatenate([np.zeros(offset, np.uint16), bits.reshape(-1)]), dtype)
        return buf[offset:].view(bits.shape)

    qd = dev(q) if which in ("both", "q") else None
    kd = dev(k) if which in ("both", "k") else None
    qo, ko = ad.qk_rmsnorm(qd, kd, dev_tensor(wq, dtype), dev_tensor(wk, dtype), 1e-6)
    torch.cuda.synchronize()
    if qd is not None:
        assert_bits_equal(host_bits(qo), oracle.qk_rmsnorm(q, Dh, wq, 1e-6, dtype, threads=THREADS)[1], dtype,
                          f"q Dh={Dh}")
    if kd is not None:
        assert_bits_equal(host_bits(ko), oracle.qk_rmsnorm(k, Dh, wk, 1e-6, dtype, threads=THREADS)[1], dtype,
                          f"k Dh={Dh}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("Dh", [4, 64, 100, 128])
def test_qk_rmsnorm(ad, Dh, dtype):
    qk_case(ad, 1003, Dh, dtype, seed=Dh)


def test_qk_rmsnorm_unaligned_dh128_and_single_tensor(ad):
    qk_case(ad, 517, 128, seed=81, offset=4)      # the one-thread-per-row kernel
    qk_case(ad, 300, 128, seed=82, which="q")
    qk_case(ad, 300, 128, seed=83, which="k")


def test_qk_rmsnorm_zimage_like_shape(ad):
    # 30 heads of 128, 4096 tokens (q and k): one launch, every row checked
    qk_case(ad, 4096 * 30, 128, seed=91)
