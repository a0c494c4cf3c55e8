"""Pins of the oracle's storage conversions against library routines.

bf16 <- f32 against torch's round-to-nearest-even conversion, fp16 <- f32
against numpy's (and, on every one of the 2^32 binary32 bit patterns, both
against torch's round-to-nearest-even conversions), and both
decodings exhaustively.  A stratified sample (every value of the upper 16
bits combined with low halves chosen to hit every rounding case: exact,
below / at / above the halfway point, odd and even) runs first as a quick
check.
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import oracle

LOW = np.array([0x0000, 0x0001, 0x0FFF, 0x1000, 0x1001, 0x17FF, 0x1800, 0x2000, 0x3000, 0x3001,
                0x4000, 0x7FFF, 0x8000, 0x8001, 0x9000, 0xBFFF, 0xC000, 0xE000, 0xEFFF, 0xF000,
                0xFFFF, 0x0800, 0x0400, 0x5A5A, 0xA5A5], dtype=np.uint32)


def stratified_f32():
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    u = (hi[:, None] | LOW[None, :]).reshape(-1)
    return u.view(np.float32)


def test_bf16_decode_exhaustive(oracle_lib):
    h = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.from16(h, "bf16")
    ref = torch.from_numpy(h.view(np.int16)).view(torch.bfloat16).float().numpy()
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


def test_fp16_decode_exhaustive(oracle_lib):
    h = np.arange(1 << 16, dtype=np.uint16)
    got = oracle.from16(h, "fp16")
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_bf16_encode_vs_torch(oracle_lib):
    f = stratified_f32()
    got = oracle.to16(f, "bf16")
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(got[nan] == 0x7FC0)


def test_fp16_encode_vs_numpy(oracle_lib):
    f = stratified_f32()
    got = oracle.to16(f, "fp16")
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(got[nan] == 0x7E00)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_roundtrip_is_identity(oracle_lib, dtype):
    h = np.arange(1 << 16, dtype=np.uint16)
    f = oracle.from16(h, dtype)
    back = oracle.to16(f, dtype)
    keep = ~np.isnan(f)
    assert np.array_equal(back[keep], h[keep])


CHUNK = 1 << 24


def _exhaustive_chunk(c):
    """Conversions of the binary32 patterns [c * CHUNK, (c + 1) * CHUNK) by the
    oracle and by the library routines: returns (mismatches, examples)."""
    u = np.arange(c * CHUNK, (c + 1) * CHUNK, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    nan = np.isnan(f)
    bad, ex = 0, []
    got = oracle.to16(f, "bf16")
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    miss = (got != ref) & ~nan
    miss |= nan & (got != 0x7FC0)
    if miss.any():
        i = np.flatnonzero(miss)
        bad += i.size
        ex += [("bf16", hex(int(u[j])), hex(int(got[j])), hex(int(ref[j]))) for j in i[:3]]
    got = oracle.to16(f, "fp16")
    ref = torch.from_numpy(f).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    miss = (got != ref) & ~nan
    miss |= nan & (got != 0x7E00)
    if miss.any():
        i = np.flatnonzero(miss)
        bad += i.size
        ex += [("fp16", hex(int(u[j])), hex(int(got[j])), hex(int(ref[j]))) for j in i[:3]]
    return bad, ex


def test_encode_every_binary32_pattern(oracle_lib):
    """All 2^32 binary32 inputs: the oracle's bf16 and fp16 equal torch's
    (every non-NaN input), and every NaN input gives the canonical quiet
    NaN."""
    n = (1 << 32) // CHUNK
    workers = max(1, min(8, os.cpu_count() or 1))
    bad, ex = 0, []
    with concurrent.futures.ThreadPoolExecutor(workers) as pool:
        for b, e in pool.map(_exhaustive_chunk, range(n)):
            bad += b
            ex += e
    assert bad == 0, (bad, ex[:8])
