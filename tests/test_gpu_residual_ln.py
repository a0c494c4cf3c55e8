"""GPU parity of adaln_residual_gate_ln_modulate (residual gate-add fused in
front of LayerNorm + adaLN modulate) with the oracle, bit for bit, through
the C ABI: both outputs, r and out."""
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


def case(ad, B, N, D, dtype="bf16", seed=0, gate_b=True, in_place=None, rows=None, eps=1e-5):
    x = synth.normal_bits(seed, B * N * D, 0, 1, dtype).reshape(B, N, D)
    y = synth.normal_bits(seed + 9, B * N * D, 0, 1, dtype).reshape(B, N, D)
    nb = B if gate_b else 1
    gsc = synth.normal_bits(seed + 1, nb * 3 * D, 0, 0.1, dtype).reshape(nb, 3, D)  # gate, scale, shift
    xg, yg, tg = dev_tensor(x, dtype), dev_tensor(y, dtype), dev_tensor(gsc, dtype)
    r_out = {"x": xg, "y": yg}.get(in_place)
    r, out = ad.residual_gate_ln_modulate(xg, tg[:, 0:1], yg, tg[:, 1:2], tg[:, 2:3], eps, r_out=r_out)
    torch.cuda.synchronize()
    srow = 3 * D if gate_b else 0
    ids, r_ref, o_ref = oracle.residual_gate_ln_modulate(x, gsc, 0, srow, y, B, N, D, gsc, D, srow, gsc,
                                                         2 * D, srow, eps, dtype, rows=rows, threads=THREADS)
    assert_bits_equal(host_bits(r).reshape(B * N, D)[ids], r_ref, dtype, f"r B={B} N={N} D={D}")
    assert_bits_equal(host_bits(out).reshape(B * N, D)[ids], o_ref, dtype, f"out B={B} N={N} D={D}")


def test_glm_shape(ad):
    case(ad, 1, 4096, 4096)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [4, 12, 512, 516, 2240, 3072, 4096])
def test_fused_kernel_shapes(ad, D, dtype):
    case(ad, 3, 37, D, dtype, seed=D)


@pytest.mark.parametrize("D", [4100, 5120, 6144, 8192])
def test_large_d(ad, D):
    # rows of up to 6144 in registers (one CTA per SM); past that the general kernel
    case(ad, 2, 19, D, seed=D + 1)


def test_broadcast_rows_and_in_place(ad):
    case(ad, 4, 33, 1024, gate_b=False, seed=3)
    case(ad, 2, 50, 2240, in_place="x", seed=4)
    case(ad, 2, 50, 2240, in_place="y", seed=5)


def test_large_batch_without_the_shared_table(ad):
    # B * D * 6 > 32 KiB: gate / scale / shift read from global memory
    case(ad, 9, 24, 1024, seed=6)


@pytest.mark.parametrize("B,D", [(2, 2728), (2, 2732), (2, 4096), (4, 1364), (4, 2048)])
def test_shared_table_size_edge(ad, B, D):
    # the gate, op and shift table takes B * D * 6 bytes: 32736 (the last
    # size kept in shared memory), then 32784, 49152, 32736, 49152
    case(ad, B, 17, D, seed=B * D)


def test_matches_the_two_ops_in_sequence(ad):
    B, N, D = 2, 64, 2048
    x = synth.normal_bits(7, B * N * D, 0, 1).reshape(B, N, D)
    y = synth.normal_bits(8, B * N * D, 0, 1).reshape(B, N, D)
    gsc = synth.normal_bits(9, B * 3 * D, 0, 0.1).reshape(B, 3, D)
    xg, yg, tg = dev_tensor(x), dev_tensor(y), dev_tensor(gsc)
    r, out = ad.residual_gate_ln_modulate(xg, tg[:, 0:1], yg, tg[:, 1:2], tg[:, 2:3], 1e-6)
    r2 = ad.residual_gate_add(xg, tg[:, 0:1], yg)
    out2 = ad.ln_modulate(r2, tg[:, 1:2], tg[:, 2:3], 1e-6)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(r), host_bits(r2))
    assert np.array_equal(host_bits(out), host_bits(out2))
