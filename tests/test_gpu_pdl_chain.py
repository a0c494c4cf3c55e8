"""All ops chained on one stream with programmatic dependent launch:
each op reads what the op before it wrote, so a kernel that read its input
before its producer finished would return wrong bits.  Every kernel lets its
dependents launch right after its own wait; the chain runs eagerly and as a
replayed CUDA graph, and every stage is compared with the same chain on the
oracle.  A second chain runs the newer kernels the same way: the
per-token-gated RMSNorm, the QK RMSNorm, the FP8 output and the table
slicer."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import THREADS, assert_bits_equal, dev_tensor, host_bits

pytestmark = pytest.mark.gpu

B, N, D, DH = 1, 512, 2048, 128


@pytest.fixture(scope="module")
def ad():
    import adaln_modulate_gb300
    assert torch.cuda.is_available()
    return adaln_modulate_gb300


@pytest.fixture(scope="module")
def chain_ref():
    x = synth.normal_bits(51, N * D, 0, 1).reshape(N, D)
    bias = synth.normal_bits(52, D, 0, 0.02)
    y = synth.normal_bits(53, N * D, 0, 1).reshape(N, D)
    gsc = synth.normal_bits(54, 3 * D, 0, 0.1)            # gate, scale, shift rows
    wq = synth.normal_bits(55, DH, 1.0, 0.05)
    bq = synth.normal_bits(56, DH, 0.0, 0.05)
    g = oracle.bias_gelu_tanh(x, bias, N, D, threads=THREADS)[1]
    r = oracle.residual_gate_add(g, gsc, 0, 0, y, B, N, D, threads=THREADS)[1]
    ln = oracle.ln_modulate(r, B, N, D, (N * D, D, 1), gsc, D, 0, gsc, 2 * D, 0, 1e-6,
                            threads=THREADS)[1]
    qk = oracle.qk_head_layernorm(ln, DH, wq, bq, 1e-6, threads=THREADS)[1]
    # r read as the transposed view of a contiguous (1, 512, 2048) tensor:
    # 2048 tokens of 512 channels (the TMA tile kernel)
    lt = oracle.ln_modulate(r, 1, D, N, (N * D, 1, D), gsc, N, 0, gsc, 2 * N, 0, 1e-6,
                            threads=THREADS)[1]
    # the fused residual gate-add + LN+modulate of g gives r and ln again
    return dict(x=x, bias=bias, y=y, gsc=gsc, wq=wq, bq=bq, g=g, r=r, ln=ln, qk=qk, lt=lt, rf=r, lf=ln)


def _chain(ad, t):
    pdl = ad.FLAG_PDL
    ad.bias_gelu_tanh(t["x"], t["bias"], out=t["g"], flags=pdl)
    rows = t["gsc"].view(3, 1, D)                       # gate, scale, shift as (1, D) rows
    ad.residual_gate_add(t["g"].view(B, N, D), rows[0], t["y"].view(B, N, D),
                         out=t["r"].view(B, N, D), flags=pdl)
    ad.ln_modulate(t["r"].view(B, N, D), rows[1], rows[2], 1e-6, out=t["ln"].view(B, N, D),
                   flags=pdl)
    ad.qk_head_layernorm(t["ln"].view(-1, DH), None, t["wq"], t["bq"], t["wq"], t["bq"], 1e-6,
                         q_out=t["qk"].view(-1, DH), flags=pdl)
    ad.residual_gate_ln_modulate(t["g"].view(B, N, D), rows[0], t["y"].view(B, N, D), rows[1], rows[2], 1e-6,
                                 r_out=t["rf"].view(B, N, D), out=t["lf"].view(B, N, D), flags=pdl)
    flat = t["gsc"].view(-1)
    ad.ln_modulate(t["r"].view(1, N, D).permute(0, 2, 1), flat[N:2 * N].view(1, N),
                   flat[2 * N:3 * N].view(1, N), 1e-6, out=t["lt"].view(1, D, N), flags=pdl)


def _tensors(ref):
    t = {k: dev_tensor(ref[k]) for k in ("x", "bias", "y", "gsc", "wq", "bq")}
    for k in ("g", "r", "ln", "qk", "lt", "rf", "lf"):
        t[k] = torch.zeros((N, D), dtype=torch.bfloat16, device="cuda")
    return t


def _check(t, ref, what):
    torch.cuda.synchronize()
    for k in ("g", "r", "ln", "qk", "lt", "rf", "lf"):
        assert_bits_equal(host_bits(t[k]).reshape(-1), ref[k].reshape(-1), what=f"{what}: {k}")


def test_chain_eager(ad, chain_ref):
    t = _tensors(chain_ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            for k in ("g", "r", "ln", "qk", "lt", "rf", "lf"):
                t[k].zero_()          # a plain kernel between the chains
            _chain(ad, t)
    s.synchronize()
    _check(t, chain_ref, "eager chain")


def test_chain_in_a_graph(ad, chain_ref):
    ad.init(torch.cuda.current_device())   # GELU tables built before capture
    t = _tensors(chain_ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _chain(ad, t)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for k in ("g", "r", "ln", "qk", "lt", "rf", "lf"):
                t[k].zero_()
            _chain(ad, t)
    for _ in range(3):
        g.replay()
    _check(t, chain_ref, "graph chain")


# a second chain through the newer kernels: GELU -> per-token-gated RMSNorm +
# modulate (per-token rows) -> QK RMSNorm -> LN + modulate into FP8, and the
# table slicer reading the QK output; every stage reads the one before it
B2, N2, D2 = 1, 256, 1024


@pytest.fixture(scope="module")
def chain2_ref():
    x = synth.normal_bits(61, N2 * D2, 0, 1).reshape(N2, D2)
    bias = synth.normal_bits(62, D2, 0, 0.02)
    y = synth.normal_bits(63, N2 * D2, 0, 1).reshape(N2, D2)
    gs = synth.normal_bits(64, N2, 0, 0.5)
    tab = synth.normal_bits(65, N2 * 6 * D2, 0, 0.1)
    w = synth.normal_bits(66, DH, 1.0, 0.05)
    sc8 = synth.normal_bits(67, 2 * D2, 0, 0.1)
    ktab = (synth.normal_bits(68, 8 * 128, 0, 0.05).astype(np.uint32) << 16).view(np.float32).reshape(8, 128)
    g = oracle.bias_gelu_tanh(x, bias, N2, D2, threads=THREADS)[1]
    _, r, o = oracle.norm_scale_shift("rms", g, B2, N2, D2, (N2 * D2, D2, 1), tab, D2, N2 * 6 * D2, 6 * D2, tab, 0,
                                      N2 * 6 * D2, 6 * D2, 1e-6, gate=(gs, 0, N2, 1, 0), y=y, threads=THREADS)
    qk = oracle.qk_rmsnorm(o, DH, w, 1e-6, threads=THREADS)[1]
    f8 = oracle.ln_modulate_fp8(qk, B2, N2, D2, (N2 * D2, D2, 1), sc8, D2, 0, sc8, 0, 0, 1e-6, 0.05,
                                threads=THREADS)[1]
    sl = oracle.temb_table_slices(ktab, "fp32", qk, "bf16", 1, N2, 8, 128)   # qk as (1, N2, 8, 128)
    return dict(x=x, bias=bias, y=y, gs=gs, tab=tab, w=w, sc8=sc8, ktab=ktab, g=g, r=r, o=o, qk=qk, f8=f8, sl=sl)


def _tensors2(ref):
    t = {k: dev_tensor(ref[k]) for k in ("x", "bias", "y", "gs", "tab", "w", "sc8")}
    t["ktab"] = torch.from_numpy(ref["ktab"]).cuda()
    t["qs"] = torch.tensor([0.05], dtype=torch.float32, device="cuda")
    for k in ("g", "r", "o", "qk"):
        t[k] = torch.zeros((N2, D2), dtype=torch.bfloat16, device="cuda")
    t["f8"] = torch.zeros((N2, D2), dtype=torch.uint8, device="cuda")
    t["sl"] = torch.zeros((8, 1, N2, 128), dtype=torch.float32, device="cuda")
    return t


def _chain2(ad, t):
    pdl = ad.FLAG_PDL
    ad.bias_gelu_tanh(t["x"], t["bias"], out=t["g"], flags=pdl)
    tab = t["tab"].view(1, N2, 6, D2)
    ad.norm_scale_shift(t["g"].view(1, N2, D2), tab[:, :, 1], tab[:, :, 0], 1e-6, norm="rms",
                        gate=t["gs"].view(1, N2, 1), y=t["y"].view(1, N2, D2), r_out=t["r"].view(1, N2, D2),
                        out=t["o"].view(1, N2, D2), flags=pdl)
    ad.qk_rmsnorm(t["o"].view(-1, DH), None, t["w"], t["w"], 1e-6, q_out=t["qk"].view(-1, DH), flags=pdl)
    sc = t["sc8"].view(1, 2, D2)
    ad.ln_modulate_fp8(t["qk"].view(1, N2, D2), sc[:, 1:2], sc[:, 0:1], 1e-6, t["qs"], out=t["f8"].view(1, N2, D2),
                       flags=pdl)
    ad.temb_table_slices(t["ktab"], t["qk"].view(1, N2, 8, 128), out=t["sl"], flags=pdl)


def _check2(t, ref, what):
    torch.cuda.synchronize()
    for k in ("g", "r", "o", "qk"):
        assert_bits_equal(host_bits(t[k]).reshape(-1), ref[k].reshape(-1), what=f"{what}: {k}")
    assert np.array_equal(t["f8"].cpu().numpy().reshape(-1), ref["f8"].reshape(-1)), f"{what}: f8"
    assert np.array_equal(t["sl"].cpu().numpy().view(np.uint32), ref["sl"].view(np.uint32)), f"{what}: slices"


def test_chain2_eager(ad, chain2_ref):
    t = _tensors2(chain2_ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            for k in ("g", "r", "o", "qk", "f8", "sl"):
                t[k].zero_()
            _chain2(ad, t)
    s.synchronize()
    _check2(t, chain2_ref, "eager chain 2")


def test_chain2_in_a_graph(ad, chain2_ref):
    ad.init(torch.cuda.current_device())
    t = _tensors2(chain2_ref)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        _chain2(ad, t)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for k in ("g", "r", "o", "qk", "f8", "sl"):
                t[k].zero_()
            _chain2(ad, t)
    for _ in range(3):
        g.replay()
    _check2(t, chain2_ref, "graph chain 2")
