"""GPU parity of adaln_qk_head_layernorm, adaln_residual_gate_add and
adaln_bias_gelu_tanh with the oracle, bit for bit, through the C ABI."""
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


# ------------------------------------------------------------------ qk

def qk_case(ad, rows_q, rows_k, Dh, dtype="bf16", in_place=False, seed=0):
    q = synth.normal_bits(seed, rows_q * Dh, 0, 2, dtype).reshape(rows_q, Dh)
    k = synth.normal_bits(seed + 8, rows_k * Dh, 0, 2, dtype).reshape(rows_k, Dh)
    wq, bq, wk, bk = (synth.normal_bits(seed + s, Dh, m, 0.05, dtype)
                      for s, m in ((3, 1.0), (4, 0.0), (5, 1.0), (6, 0.0)))
    qg = dev_tensor(q, dtype) if rows_q else None
    kg = dev_tensor(k, dtype) if rows_k else None
    ws = [dev_tensor(v, dtype) for v in (wq, bq, wk, bk)]
    qo, ko = ad.qk_head_layernorm(qg, kg, *ws, 1e-6, q_out=qg if in_place else None,
                                  k_out=kg if in_place else None)
    torch.cuda.synchronize()
    if rows_q:
        ref = oracle.qk_head_layernorm(q, Dh, wq, bq, 1e-6, dtype, threads=THREADS)[1]
        assert_bits_equal(host_bits(qo), ref, dtype, f"q rows={rows_q} Dh={Dh}")
    if rows_k:
        ref = oracle.qk_head_layernorm(k, Dh, wk, bk, 1e-6, dtype, threads=THREADS)[1]
        assert_bits_equal(host_bits(ko), ref, dtype, f"k rows={rows_k} Dh={Dh}")


def test_qk_glm_full(ad):
    rows = 4360 * 32
    qk_case(ad, rows, rows, 128)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("Dh", [4, 8, 64, 100, 124, 128])
def test_qk_shapes(ad, Dh, dtype):
    qk_case(ad, 1001, 333, Dh, dtype, seed=Dh)


def test_qk_one_tensor_and_in_place(ad):
    qk_case(ad, 0, 257, 128)
    qk_case(ad, 259, 0, 64)
    qk_case(ad, 1003, 997, 128, in_place=True)


# ------------------------------------------------------------- gate add

def gate_case(ad, B, N, D, dtype="bf16", gate_rows=None, in_place=False, seed=0):
    x = synth.normal_bits(seed, B * N * D, 0, 1, dtype).reshape(B, N, D)
    y = synth.normal_bits(seed + 9, B * N * D, 0, 1, dtype).reshape(B, N, D)
    g = synth.normal_bits(seed + 10, B * 3 * D, 0, 0.1, dtype).reshape(B, 3, D)   # chunk 2 of a table
    xg, yg = dev_tensor(x, dtype), dev_tensor(y, dtype)
    gg = dev_tensor(g, dtype)[:, 2:3]
    out = ad.residual_gate_add(xg, gg, yg, out=xg if in_place else None)
    torch.cuda.synchronize()
    ref = oracle.residual_gate_add(x, g, 2 * D, 3 * D, y, B, N, D, dtype, threads=THREADS)[1]
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref, dtype, f"gate {B},{N},{D}")


def test_gate_glm_full(ad):
    gate_case(ad, 1, 4096, 4096)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [1, 3, 4, 8, 12, 16, 100, 2240, 3072, 4097])
def test_gate_shapes(ad, D, dtype):
    gate_case(ad, 2, 37, D, dtype, seed=D)


def test_gate_in_place(ad):
    gate_case(ad, 2, 100, 1024, in_place=True)


# ----------------------------------------------------------- bias + GELU

@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gelu_every_input_pattern(ad, dtype):
    # x runs over all 65536 patterns with bias 0: out = table[round(x + 0)]
    x = np.arange(1 << 16, dtype=np.uint16).reshape(64, 1024)
    bias = np.zeros(1024, dtype=np.uint16)
    out = ad.bias_gelu_tanh(dev_tensor(x, dtype), dev_tensor(bias, dtype))
    ref = oracle.bias_gelu_tanh(x, bias, 64, 1024, dtype)[1]
    assert_bits_equal(host_bits(out), ref, dtype, "all patterns")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gelu_wan_full(ad, dtype):
    w = synth.gelu_wan(dtype)
    rows, width = 32760, 13824
    x = w.tensors["x"].draw(dtype)
    bias = w.tensors["bias"].draw(dtype)
    out = ad.bias_gelu_tanh(dev_tensor(x, dtype), dev_tensor(bias, dtype))
    got = host_bits(out)
    del out
    # the whole output, all 32760 x 13824 elements, against the oracle
    ids, ref = oracle.bias_gelu_tanh(x, bias, rows, width, dtype, threads=THREADS)
    assert ids.size == rows
    assert_bits_equal(got, ref, dtype, f"wan {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("width", [1, 3, 4, 8, 12, 16, 1000, 13824, 13825])
def test_gelu_widths(ad, width, dtype):
    rows = 37
    x = synth.normal_bits(width, rows * width, 0, 3, dtype).reshape(rows, width)
    bias = synth.normal_bits(width + 1, width, 0, 0.5, dtype)
    out = ad.bias_gelu_tanh(dev_tensor(x, dtype), dev_tensor(bias, dtype))
    ref = oracle.bias_gelu_tanh(x, bias, rows, width, dtype)[1]
    assert_bits_equal(host_bits(out), ref, dtype, f"width {width}")


def test_gelu_in_place(ad):
    x = synth.normal_bits(1, 64 * 2048, 0, 1).reshape(64, 2048)
    bias = synth.normal_bits(2, 2048, 0, 0.02)
    xg = dev_tensor(x)
    ad.bias_gelu_tanh(xg, dev_tensor(bias), out=xg)
    assert_bits_equal(host_bits(xg), oracle.bias_gelu_tanh(x, bias, 64, 2048)[1], what="in place")
