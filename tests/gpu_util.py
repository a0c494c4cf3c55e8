"""Helpers of the GPU parity tests: move 16-bit patterns between numpy and
CUDA tensors and compare GPU outputs with the oracle bit for bit."""
import os

import numpy as np
import torch

TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}
THREADS = max(1, min(16, os.cpu_count() or 1))


def dev_tensor(bits, dtype="bf16"):
    bits = np.ascontiguousarray(bits)
    return torch.from_numpy(bits.view(np.int16)).view(TORCH_DT[dtype]).cuda()


def host_bits(t):
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def is_nan16(bits, dtype="bf16"):
    b = np.asarray(bits, dtype=np.uint16)
    if dtype == "bf16":
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    return ((b & 0x7C00) == 0x7C00) & ((b & 0x03FF) != 0)


def assert_bits_equal(got, ref, dtype="bf16", what=""):
    """Bit-exact, except that a NaN matches any NaN (payloads unspecified)."""
    got = np.asarray(got, dtype=np.uint16).reshape(-1)
    ref = np.asarray(ref, dtype=np.uint16).reshape(-1)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    gn, rn = is_nan16(got, dtype), is_nan16(ref, dtype)
    bad = (gn != rn) | (~gn & (got != ref))
    if bad.any():
        idx = np.nonzero(bad)[0]
        sample = [(int(i), hex(int(got[i])), hex(int(ref[i]))) for i in idx[:8]]
        raise AssertionError(f"{what}: {idx.size} of {got.size} elements differ, e.g. {sample}")
