"""The allocation-free bias + tanh-GELU entry point, called through the C ABI.

adaln_bias_gelu_tanh_noalloc is for callers that cannot let a library
allocate device memory: a process whose memory pool owns the whole GPU,
code that must not hit the implicit synchronisation of cudaMalloc /
cudaFree, or a program that forbids allocations after start-up.  It keeps
its lookup tables in a fixed array of the library's device image instead of
allocating them, and must return exactly what adaln_bias_gelu_tanh returns.

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.  It also passes on its own in a
fresh process (its first call then does the one-time table set-up).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import TORCH_DT, assert_bits_equal, dev_tensor, host_bits

pytestmark = pytest.mark.gpu

CODE = {"bf16": 0, "fp16": 1}


def _call(fn, out, x, bias, rows, width, dtype):
    stream = torch.cuda.current_stream().cuda_stream
    return fn(out.data_ptr(), x.data_ptr(), bias.data_ptr(), rows, width, CODE[dtype], 0, stream)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_noalloc_matches_the_allocating_entry_point_on_two_calls(dtype):
    import adaln_modulate_gb300 as ad

    rows, width = 257, 13824
    for call, seed in enumerate((41, 42)):  # two calls in a row, different inputs
        x = synth.normal_bits(seed, rows * width, 0, 1.5, dtype).reshape(rows, width)
        bias = synth.normal_bits(seed + 100, width, 0, 0.02, dtype)
        xg, bg = dev_tensor(x, dtype), dev_tensor(bias, dtype)
        ref = torch.empty((rows, width), dtype=TORCH_DT[dtype], device="cuda")
        got = torch.full((rows, width), 7.0, dtype=TORCH_DT[dtype], device="cuda")
        st_na = _call(ad.capi.adaln_bias_gelu_tanh_noalloc, got, xg, bg, rows, width, dtype)
        st_ref = _call(ad.capi.adaln_bias_gelu_tanh, ref, xg, bg, rows, width, dtype)
        torch.cuda.synchronize()
        assert st_na == 0 and st_ref == 0, (st_na, st_ref)
        assert_bits_equal(host_bits(got), host_bits(ref), dtype, f"noalloc call {call} vs allocating")
        if call == 0:  # and both against the CPU oracle on a few rows
            ids, want = oracle.bias_gelu_tanh(x, bias, rows, width, dtype, rows=[0, 100, 256])
            assert_bits_equal(host_bits(got)[ids], want, dtype, "noalloc vs oracle")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_noalloc_every_input_pattern(dtype):
    import adaln_modulate_gb300 as ad

    x = np.arange(1 << 16, dtype=np.uint16).reshape(64, 1024)
    bias = np.zeros(1024, dtype=np.uint16)
    xg, bg = dev_tensor(x, dtype), dev_tensor(bias, dtype)
    got = torch.empty((64, 1024), dtype=TORCH_DT[dtype], device="cuda")
    assert _call(ad.capi.adaln_bias_gelu_tanh_noalloc, got, xg, bg, 64, 1024, dtype) == 0
    torch.cuda.synchronize()
    assert_bits_equal(host_bits(got), oracle.bias_gelu_tanh(x, bias, 64, 1024, dtype)[1], dtype,
                      "all patterns")


def test_noalloc_rejects_bad_arguments_without_launching():
    import adaln_modulate_gb300 as ad

    f = ad.capi.adaln_bias_gelu_tanh_noalloc
    assert f(1 << 40, 1 << 41, 1 << 42, 0, 16, 0, 0, None) == 3      # no rows
    assert f(1 << 40, 1 << 41, 1 << 42, 4, 16, 7, 0, None) == 2      # unknown storage type
    assert f(1 << 40, 1 << 40, 1 << 40, 4, 16, 0, 0, None) == 7      # bias overlaps out
