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
import os
import subprocess
import sys
import textwrap

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


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _fresh_process(body):
    """Runs body in a new Python process (so the entry point's one-time table
    set-up has not happened yet) and returns its stdout."""
    code = textwrap.dedent("""
        import sys
        sys.path.insert(0, {root!r})
        sys.path.insert(0, {tests!r})
        import numpy as np
        import torch
        import adaln_modulate_gb300 as ad
        import synth
        from gpu_util import TORCH_DT, dev_tensor, host_bits
        CODE = {{"bf16": 0, "fp16": 1}}
    """).format(root=ROOT, tests=os.path.join(ROOT, "tests")) + textwrap.dedent(body)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    return r.stdout


def test_noalloc_first_call_inside_a_capture_is_refused_and_the_capture_survives():
    # The first call on a device sets up its table on the caller's stream and
    # waits for it; inside a stream capture that would break the caller's
    # graph, so the call must return ADALN_E_CUDA with a message, launch
    # nothing and leave the capture valid.  After the capture, a plain first
    # call works.
    out = _fresh_process("""
        rows, width = 8, 1024
        x = torch.randn(rows, width, device="cuda").to(torch.bfloat16)
        b = torch.zeros(width, device="cuda", dtype=torch.bfloat16)
        o = torch.empty_like(x)
        y = torch.zeros(16, device="cuda")
        s = torch.cuda.Stream()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            y.add_(1)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            st = ad.capi.adaln_bias_gelu_tanh_noalloc(o.data_ptr(), x.data_ptr(), b.data_ptr(), rows, width,
                                                      0, 0, s.cuda_stream)
            y.add_(1)
        msg = ad.capi.adaln_last_cuda_error().decode()
        g.replay()
        torch.cuda.synchronize()
        assert st == 8, st
        assert "before capturing" in msg, msg
        assert float(y[0]) == 2.0, float(y[0])        # the captured work ran: the capture stayed valid
        st2 = ad.capi.adaln_bias_gelu_tanh_noalloc(o.data_ptr(), x.data_ptr(), b.data_ptr(), rows, width, 0, 0,
                                                   torch.cuda.current_stream().cuda_stream)
        ref = torch.empty_like(x)
        st3 = ad.capi.adaln_bias_gelu_tanh(ref.data_ptr(), x.data_ptr(), b.data_ptr(), rows, width, 0, 0,
                                           torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert st2 == 0 and st3 == 0, (st2, st3)
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16))
        print("ok")
    """)
    assert out.strip().endswith("ok")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_noalloc_first_call_is_ordered_after_work_on_its_stream(dtype):
    # Work queued on the caller's stream before the first call (a slow kernel,
    # then the copy that writes the real input) must finish before the table
    # set-up and the GELU read x: the output equals the allocating entry
    # point's on the final input, not on the stale one.
    out = _fresh_process("""
        dtype = {dtype!r}
        rows, width = 64, 2048
        xb = synth.normal_bits(5, rows * width, 0, 1.5, dtype).reshape(rows, width)
        bb = synth.normal_bits(6, width, 0, 0.02, dtype)
        real, b = dev_tensor(xb, dtype), dev_tensor(bb, dtype)
        x = torch.zeros_like(real)                       # stale contents until the side stream writes it
        o = torch.empty_like(real)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            torch.cuda._sleep(50_000_000)                # tens of ms on the side stream
            x.copy_(real)
            st = ad.capi.adaln_bias_gelu_tanh_noalloc(o.data_ptr(), x.data_ptr(), b.data_ptr(), rows, width,
                                                      CODE[dtype], 0, side.cuda_stream)
        torch.cuda.synchronize()
        ref = torch.empty_like(real)
        st2 = ad.capi.adaln_bias_gelu_tanh(ref.data_ptr(), real.data_ptr(), b.data_ptr(), rows, width,
                                           CODE[dtype], 0, torch.cuda.current_stream().cuda_stream)
        torch.cuda.synchronize()
        assert st == 0 and st2 == 0, (st, st2)
        assert np.array_equal(host_bits(o), host_bits(ref))
        print("ok")
    """.format(dtype=dtype))
    assert out.strip().endswith("ok")
