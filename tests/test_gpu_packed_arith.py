"""Every modulate, gate and bias step on the GPU adds or multiplies two
16-bit storage values with one packed instruction (add.rn / mul.rn on bf16x2
or f16x2).  The chains specify binary32 arithmetic followed by one rounding
to the storage type (PR #34015, "实现拆解" 2: the pass-2 rounding points;
PR #34008 "实现拆解" 3 for the gate; PR #37075 "关键源码片段" for the bias).
Double rounding is innocuous here (binary32 has at least 2p + 2 significand
bits for p = 8 and 11), and this test checks it instead of relying on the
theorem: all 2^32 operand pairs, for both operations and both storage types,
against binary32 arithmetic and a round-to-nearest-even conversion written
from the IEEE definition in integer arithmetic (NaN compared as NaN).  The
hardware conversion cvt.rn is checked against that rounding on the same
binary32 values."""
import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    so = str(tmp_path_factory.mktemp("packed") / "packed_sweep.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-fmad=false", "-shared", os.path.join(HERE, "cuda", "packed_sweep.cu"), "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.packed_sweep.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    return lib


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("op", ["add", "mul"])
def test_every_operand_pair(helper, op, dtype):
    out = (ctypes.c_ulonglong * 3)()
    assert helper.packed_sweep(int(op == "mul"), int(dtype == "fp16"), out) == 0
    bad, bad_cvt, first = out[0], out[1], out[2]
    assert bad == 0, f"{op} {dtype}: {bad} of 2^32 pairs differ, first a={first >> 16:#06x} b={first & 0xFFFF:#06x}"
    assert bad_cvt == 0, f"{op} {dtype}: cvt.rn differs from the IEEE rounding on {bad_cvt} results"
