"""Pins of the oracle's temb_table_slices (no GPU).

The op is one IEEE binary32 addition per element of two exactly promoted
operands, so numpy's float32 addition of the same operands (promoted by
numpy's own bf16 / fp16 decoding) fixes every output bit; the pins also
fix the slice order (chunk k of the temb row goes to slice k), the
broadcast of the table over (b, s) and the signed-zero and non-finite
cases of the addition."""
import numpy as np
import pytest

import oracle
import synth
from fp64ref import value16


def _np_value(a, dt):
    return a.astype(np.float32) if dt == "fp32" else value16(a, dt).astype(np.float32)


@pytest.mark.parametrize("table_dt,temb_dt", [("fp32", "bf16"), ("bf16", "bf16"), ("fp32", "fp32"),
                                              ("fp16", "fp16"), ("bf16", "fp32")])
def test_slices_equal_numpy_binary32_add(oracle_lib, table_dt, temb_dt):
    B, S, K, D = 2, 5, 6, 72

    def draw(seed, n, std, dt):
        if dt == "fp32":
            return (np.random.default_rng(seed).standard_normal(n) * std).astype(np.float32)
        return synth.normal_bits(seed, n, 0, std, dt)

    table = draw(1, K * D, 0.05, table_dt).reshape(K, D)
    temb = draw(2, B * S * K * D, 1.0, temb_dt).reshape(B, S, K, D)
    out = oracle.temb_table_slices(table, table_dt, temb, temb_dt, B, S, K, D)
    ref = _np_value(table, table_dt)[None, None] + _np_value(temb, temb_dt)      # (B, S, K, D)
    assert np.array_equal(out.view(np.uint32), np.ascontiguousarray(ref.transpose(2, 0, 1, 3)).view(np.uint32))


def test_slice_order_and_broadcast(oracle_lib):
    # temb = 0 everywhere: every slice k is table row k repeated over (b, s)
    B, S, K, D = 3, 4, 6, 16
    table = np.arange(K * D, dtype=np.float32).reshape(K, D)
    out = oracle.temb_table_slices(table, "fp32", np.zeros((B, S, K, D), np.float32), "fp32", B, S, K, D)
    for k in range(K):
        assert np.array_equal(out[k], np.broadcast_to(table[k], (B, S, D)))
    # table = 0: slice k of token (b, s) is temb[b, s, k]
    temb = np.arange(B * S * K * D, dtype=np.float32).reshape(B, S, K, D)
    out = oracle.temb_table_slices(np.zeros((K, D), np.float32), "fp32", temb, "fp32", B, S, K, D)
    assert np.array_equal(out, temb.transpose(2, 0, 1, 3))


def test_signed_zero_and_non_finite(oracle_lib):
    table = np.array([[-0.0, -0.0, np.inf, 1.0, 3.0e38, -np.inf, np.nan, 2.0 ** -149]], np.float32)
    temb = np.array([[[[-0.0, 0.0, -np.inf, -1.0, 3.0e38, 1.0, 1.0, 2.0 ** -149]]]], np.float32)
    out = oracle.temb_table_slices(table, "fp32", temb, "fp32", 1, 1, 1, 8)[0, 0, 0]
    assert np.signbit(out[0]) and out[0] == 0 and not np.signbit(out[1])
    assert np.isnan(out[2]) and out[3] == 0 and not np.signbit(out[3])
    assert out[4] == np.inf and out[5] == -np.inf and np.isnan(out[6]) and out[7] == 2.0 ** -148
