"""GPU parity of adaln_ln_modulate with the oracle, bit for bit, through the
C ABI: the workloads of the pages at full size, every kernel path (rows,
tokens, general strides) on ragged shapes, fp16, in place, output guards,
non-finite inputs and programmatic dependent launch."""
import numpy as np
import pytest
import torch

import oracle
import synth
from fp64ref import bits16, ln_modulate_fp64, ulp_diff, value16
from gpu_util import THREADS, assert_bits_equal, dev_tensor, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ad():
    import adaln_modulate_gb300
    assert torch.cuda.is_available()
    return adaln_modulate_gb300


def run_both(ad, xbase, B, N, D, strides, table, sc_off, sh_off, srow, eps, dtype="bf16",
             expect=None, rows=None):
    """GPU through the C ABI on the view `strides` of xbase, and the oracle."""
    xg = dev_tensor(xbase, dtype)
    xv = torch.as_strided(xg, (B, N, D), strides)
    tg = dev_tensor(table, dtype).reshape(-1)
    sc = torch.as_strided(tg, (B, 1, D), (srow, D, 1), sc_off)
    sh = torch.as_strided(tg, (B, 1, D), (srow, D, 1), sh_off)
    if expect:
        got_variant = ad.ln_modulate_variant(xv, sc, sh, eps)
        # "tokens" / "rows": either kernel of that layout
        assert got_variant == expect or got_variant == expect + "_tma", got_variant
    out = ad.ln_modulate(xv, sc, sh, eps)
    torch.cuda.synchronize()
    ids, ref = oracle.ln_modulate(xbase, B, N, D, strides, table, sc_off, srow, table, sh_off, srow,
                                  eps, dtype, rows=rows, threads=THREADS)
    got = host_bits(out).reshape(B * N, D)[ids]
    return got, ref


# -------------------------------------------------- the pages' workloads

def test_tiny_config(ad):
    w = synth.ln_tiny()
    x, sc, sh = (w.tensors[k].draw() for k in ("x", "scale", "shift"))
    table = np.concatenate([sc.reshape(-1), sh.reshape(-1)])
    got, ref = run_both(ad, x, 1, 64, 512, (64 * 512, 512, 1), table, 0, 512, 1024, 1e-6, expect="rows")
    assert_bits_equal(got, ref, what="tiny")


@pytest.mark.parametrize("nmod,scale_chunk", [(6, 1), (2, 1), (6, 5)])
def test_sana_transposed(ad, nmod, scale_chunk):
    w = synth.ln_sana(nmod=nmod, scale_chunk=scale_chunk)
    B, N, D = 2, 1024, 2240
    x = w.tensors["x"].draw()                     # contiguous (B, D, N)
    table = w.tensors["table"].draw()             # (B, nmod, D)
    got, ref = run_both(ad, x, B, N, D, (D * N, 1, N), table, scale_chunk * D, 0, nmod * D, 1e-6,
                        expect="tokens")
    assert_bits_equal(got, ref, what=f"sana nmod={nmod} chunk={scale_chunk}")


def test_sana_transposed_sigma4_and_fp64(ad):
    B, N, D = 2, 1024, 2240
    x = synth.normal_bits(0, B * D * N, 0, 4).reshape(B, D, N)
    table = synth.normal_bits(1, B * 6 * D, 0, 0.1).reshape(B, 6, D)
    got, ref = run_both(ad, x, B, N, D, (D * N, 1, N), table, D, 0, 6 * D, 1e-6, expect="tokens")
    assert_bits_equal(got, ref, what="sana sigma 4")
    # the fp64-statistics chain: >= 99.99 % within one ulp
    xr = value16(np.ascontiguousarray(x.transpose(0, 2, 1))).reshape(B, N, D)
    for b in range(B):
        r64 = bits16(ln_modulate_fp64(xr[b], value16(table[b, 1]), value16(table[b, 0]), 1e-6))
        d = ulp_diff(got[b * N:(b + 1) * N], r64)
        assert (d <= 1).mean() >= 0.9999


@pytest.mark.parametrize("shape", [(2, 1024, 2240), (1, 37, 2240)])
def test_sana_contiguous(ad, shape):
    B, N, D = shape
    x = synth.normal_bits(0, B * N * D, 0, 4).reshape(B, N, D)
    table = synth.normal_bits(1, B * 6 * D, 0, 0.1).reshape(B, 6, D)
    got, ref = run_both(ad, x, B, N, D, (N * D, D, 1), table, 5 * D, 0, 6 * D, 1e-6, expect="rows")
    assert_bits_equal(got, ref, what=f"sana contiguous {shape}")


def test_glm_full(ad):
    w = synth.ln_glm()
    x, sc, sh = (w.tensors[k].draw() for k in ("x", "scale", "shift"))
    table = np.concatenate([sc.reshape(-1), sh.reshape(-1)])
    got, ref = run_both(ad, x, 1, 4096, 4096, (4096 * 4096, 4096, 1), table, 0, 4096, 8192, 1e-5,
                        expect="rows")
    assert_bits_equal(got, ref, what="glm")
    r64 = bits16(ln_modulate_fp64(value16(x[0]), value16(sc[0, 0]), value16(sh[0, 0]), 1e-5))
    assert (ulp_diff(got, r64) <= 1).mean() >= 0.9999


# --------------------------------------------------- every path, ragged

D_LIST = [4, 8, 12, 60, 500, 512, 516, 1020, 1536, 2240, 2244, 3072, 4096]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", D_LIST)
def test_rows_path_ragged(ad, D, dtype):
    B, N = 3, 67
    x = synth.normal_bits(D, B * N * D, 0.5, 2, dtype).reshape(B, N, D)
    table = synth.normal_bits(D + 1, B * 2 * D, 0, 0.1, dtype).reshape(B, 2, D)
    got, ref = run_both(ad, x, B, N, D, (N * D, D, 1), table, D, 0, 2 * D, 1e-6, dtype)
    assert_bits_equal(got, ref, dtype, f"rows D={D}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D,N", [(4, 8), (12, 13), (500, 67), (512, 5), (516, 9), (2240, 67),
                                 (2244, 16), (4096, 24), (6144, 9)])
def test_tokens_path_ragged(ad, D, N, dtype):
    B = 2
    x = synth.normal_bits(D + 7, B * D * N, 0, 1, dtype).reshape(B, D, N)
    table = synth.normal_bits(D + 8, B * 6 * D, 0, 0.1, dtype).reshape(B, 6, D)
    got, ref = run_both(ad, x, B, N, D, (D * N, 1, N), table, D, 0, 6 * D, 1e-6, dtype,
                        expect="tokens" if N % 8 == 0 else None)
    assert_bits_equal(got, ref, dtype, f"tokens D={D} N={N}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,N,D", [(3, 2056, 2240),   # 387 tiles of 16: several per CTA, ragged last
                                   (1, 4000, 1024),   # one sample, D % 512 == 0
                                   (2, 48, 5120),     # the largest D of the 16-token TMA tile
                                   (2, 16, 5632)])    # past it (if shared memory allows)
def test_tokens_tiles_many_per_cta(ad, B, N, D, dtype):
    x = synth.normal_bits(D + 11, B * D * N, 0.25, 1.5, dtype).reshape(B, D, N)
    table = synth.normal_bits(D + 12, B * 6 * D, 0, 0.1, dtype).reshape(B, 6, D)
    got, ref = run_both(ad, x, B, N, D, (D * N, 1, N), table, D, 0, 6 * D, 1e-6, dtype, expect="tokens")
    assert_bits_equal(got, ref, dtype, f"tokens tiles B={B} N={N} D={D}")
    assert ad.tma_wait_timeouts() == 0


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("B,N,D", [(2, 1024, 2240),   # the headline: 128 tiles, one per CTA
                                   (1, 1000, 2240),   # ragged last tile (8 of 16 tokens)
                                   (2, 40, 516),      # tail chunk, few tiles
                                   (2, 2600, 1024),   # 326 tiles: two or three per CTA
                                   (3, 1624, 512),    # ragged last tile of each sample
                                   (1, 8, 5120)])     # one half tile of the largest D
def test_tma_tile_shapes(ad, B, N, D, dtype):
    # the path needs N % 8 == 0 (16-byte d-row strides for the tensor map)
    x = synth.normal_bits(N + D, B * D * N, 0.1, 1.2, dtype).reshape(B, D, N)
    table = synth.normal_bits(N + D + 1, B * 6 * D, 0, 0.1, dtype).reshape(B, 6, D)
    got, ref = run_both(ad, x, B, N, D, (D * N, 1, N), table, D, 0, 6 * D, 1e-6, dtype, expect="tokens_tma")
    assert_bits_equal(got, ref, dtype, f"tma tiles B={B} N={N} D={D}")
    assert ad.tma_wait_timeouts() == 0


def test_sana_takes_the_tma_tile_kernel(ad):
    # the transposed headline shape goes through the TMA tiles; the largest
    # D past them through the cp.async tiles
    B, N, D = 2, 1024, 2240
    x = synth.normal_bits(35, B * D * N, 0, 1).reshape(B, D, N)
    table = synth.normal_bits(36, B * 6 * D, 0, 0.1).reshape(B, 6, D)
    got, ref = run_both(ad, x, B, N, D, (D * N, 1, N), table, D, 0, 6 * D, 1e-6,
                        expect="tokens_tma")
    assert_bits_equal(got, ref, what="tma tiles")
    xg = torch.empty((1, 6144, 16), dtype=torch.bfloat16, device="cuda")
    tg = torch.zeros((1, 2, 6144), dtype=torch.bfloat16, device="cuda")
    assert ad.ln_modulate_variant(xg.permute(0, 2, 1), tg[:, 1:2], tg[:, 0:1], 1e-6) == "tokens"


def test_tokens_pdl_orders_after_producer(ad):
    B, N, D = 2, 1024, 2240
    x = synth.normal_bits(33, B * D * N, 0, 1).reshape(B, D, N)
    table = synth.normal_bits(34, B * 6 * D, 0, 0.1).reshape(B, 6, D)
    _, ref = oracle.ln_modulate(x, B, N, D, (D * N, 1, N), table, D, 6 * D, table, 0, 6 * D, 1e-6,
                                threads=THREADS)
    s = torch.cuda.Stream()
    xg = torch.zeros((B, D, N), dtype=torch.bfloat16, device="cuda")
    src = dev_tensor(x)
    tg = dev_tensor(table)
    with torch.cuda.stream(s):
        for _ in range(3):
            xg.copy_(src)           # producer kernel on the same stream
            out = ad.ln_modulate(xg.permute(0, 2, 1), tg[:, 1:2], tg[:, 0:1], 1e-6, flags=ad.FLAG_PDL)
            xg.zero_()
    s.synchronize()
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref, what="tokens pdl")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D", [4, 516, 2240, 4100, 8192, 13824])
def test_generic_path(ad, D, dtype):
    B, N = 2, 5
    # every element at stride 3: neither rows nor tokens are contiguous
    base = synth.normal_bits(D + 9, 3 * B * N * D, 0, 1, dtype)
    table = synth.normal_bits(D + 10, B * 2 * D, 0, 0.1, dtype).reshape(B, 2, D)
    got, ref = run_both(ad, base, B, N, D, (3 * N * D, 3 * D, 3), table, 0, D, 2 * D, 1e-5, dtype,
                        expect="generic")
    assert_bits_equal(got, ref, dtype, f"generic D={D}")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("D,expect", [(4100, "rows"), (4608, "rows"), (5120, "rows"), (5632, "rows"),
                                      (6140, "rows"), (6144, "rows"), (6148, "generic")])
def test_large_contiguous_rows(ad, D, expect, dtype):
    # one CTA per SM holds rows of up to 6144 elements; past that the general kernel
    B, N = 2, 33
    x = synth.normal_bits(D + 3, B * N * D, 0, 1, dtype).reshape(B, N, D)
    table = synth.normal_bits(D + 4, B * 2 * D, 0, 0.1, dtype).reshape(B, 2, D)
    got, ref = run_both(ad, x, B, N, D, (N * D, D, 1), table, D, 0, 2 * D, 1e-6, dtype, expect=expect)
    assert_bits_equal(got, ref, dtype, what=f"D={D}")


# ------------------------------------------------------------ edge cases

def test_in_place_and_guards(ad):
    B, N, D = 2, 50, 2240
    x = synth.normal_bits(5, B * N * D, 0, 1).reshape(B, N, D)
    table = synth.normal_bits(6, B * 6 * D, 0, 0.1).reshape(B, 6, D)
    _, ref = oracle.ln_modulate(x, B, N, D, (N * D, D, 1), table, D, 6 * D, table, 0, 6 * D, 1e-6)
    tg = dev_tensor(table).reshape(-1)
    sc = torch.as_strided(tg, (B, 1, D), (6 * D, D, 1), D)
    sh = torch.as_strided(tg, (B, 1, D), (6 * D, D, 1), 0)
    # in place
    xg = dev_tensor(x)
    ad.ln_modulate(xg, sc, sh, 1e-6, out=xg)
    assert_bits_equal(host_bits(xg).reshape(B * N, D), ref, what="in place")
    # output in the middle of a guarded buffer (4 KiB of canaries each side)
    g = 2048
    buf = torch.full((B * N * D + 2 * g,), -7.25, dtype=torch.bfloat16, device="cuda")
    out = buf[g:g + B * N * D].view(B, N, D)
    ad.ln_modulate(dev_tensor(x), sc, sh, 1e-6, out=out)
    hb = host_bits(buf)
    canary = host_bits(torch.tensor([-7.25], dtype=torch.bfloat16))[0]
    assert np.all(hb[:g] == canary) and np.all(hb[-g:] == canary)
    assert_bits_equal(hb[g:-g].reshape(B * N, D), ref, what="guarded")


def test_non_finite_and_degenerate_rows(ad):
    B, N, D = 1, 6, 1024
    x = synth.normal_bits(11, B * N * D, 0, 1).reshape(B, N, D).copy()
    x[0, 0, 5] = 0x7F80          # +inf -> the whole row is NaN
    x[0, 1, 7] = 0x7FC1          # NaN
    x[0, 2, :] = 0x3FC0          # constant row: mean = 1.5, m2 = 0, y = 0
    x[0, 3, :] = 0x0001          # smallest subnormal everywhere
    x[0, 4, ::2] = 0x7F7F        # huge values: variance overflows to inf
    table = synth.normal_bits(12, 2 * D, 0, 0.1).reshape(1, 2, D).copy()
    table[0, 0, :3] = [0x0001, 0x8001, 0x8000]    # subnormal and -0 shifts
    table[0, 1, 3:6] = [0x0001, 0x807F, 0xBF80]   # subnormal scales, scale = -1
    for eps in (1e-6, 0.0):
        got, ref = run_both(ad, x, B, N, D, (N * D, D, 1), table, D, 0, 2 * D, eps)
        assert_bits_equal(got, ref, what=f"non-finite eps={eps}")


def test_pdl_flag_orders_after_producer(ad):
    B, N, D = 1, 256, 4096
    x = synth.normal_bits(13, B * N * D, 0, 1).reshape(B, N, D)
    table = synth.normal_bits(14, 2 * D, 0, 0.1).reshape(1, 2, D)
    _, ref = oracle.ln_modulate(x, B, N, D, (N * D, D, 1), table, D, 2 * D, table, 0, 2 * D, 1e-6)
    s = torch.cuda.Stream()
    xg = torch.zeros((B, N, D), dtype=torch.bfloat16, device="cuda")
    src = dev_tensor(x)
    tg = dev_tensor(table).reshape(1, 2, D)
    with torch.cuda.stream(s):
        for _ in range(3):
            xg.copy_(src)           # producer kernel on the same stream
            out = ad.ln_modulate(xg, tg[:, 1:2], tg[:, 0:1], 1e-6, flags=ad.FLAG_PDL)
            xg.zero_()
    s.synchronize()
    assert_bits_equal(host_bits(out).reshape(N, D), ref, what="pdl")


def test_broadcast_scale_and_shift_rows(ad):
    # scale / shift shared by every sample (batch stride 0)
    B, N, D = 3, 20, 768
    x = synth.normal_bits(15, B * N * D, 0, 1).reshape(B, N, D)
    table = synth.normal_bits(16, 2 * D, 0, 0.1)
    xg, tg = dev_tensor(x), dev_tensor(table)
    sc = tg[D:].view(1, 1, D).expand(B, 1, D)
    sh = tg[:D].view(1, 1, D).expand(B, 1, D)
    out = ad.ln_modulate(xg, sc, sh, 1e-6)
    _, ref = oracle.ln_modulate(x, B, N, D, (N * D, D, 1), table, D, 0, table, 0, 0, 1e-6)
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref, what="broadcast rows")


@pytest.mark.parametrize("D", [512, 2240, 4096])
def test_rows_path_with_8_byte_aligned_rows(ad, D):
    # x starts 8 bytes past a 16-byte boundary: the rows kernel's 8-byte
    # accesses only need 8-byte aligned rows
    B, N = 2, 40
    x = synth.normal_bits(D + 21, B * N * D, 0, 1).reshape(B, N, D)
    table = synth.normal_bits(D + 22, B * 2 * D, 0, 0.1).reshape(B, 2, D)
    buf = torch.empty(B * N * D + 4, dtype=torch.bfloat16, device="cuda")
    xv = buf[4:].view(B, N, D)
    xv.copy_(dev_tensor(x))
    assert xv.data_ptr() % 16 == 8
    tg = dev_tensor(table).reshape(-1)
    sc = torch.as_strided(tg, (B, 1, D), (2 * D, D, 1), D)
    sh = torch.as_strided(tg, (B, 1, D), (2 * D, D, 1), 0)
    assert ad.ln_modulate_variant(xv, sc, sh, 1e-6) == "rows"
    out = ad.ln_modulate(xv, sc, sh, 1e-6)
    _, ref = oracle.ln_modulate(x, B, N, D, (N * D, D, 1), table, D, 2 * D, table, 0, 2 * D, 1e-6)
    assert_bits_equal(host_bits(out).reshape(B * N, D), ref, what=f"8-byte aligned rows D={D}")


@pytest.mark.parametrize("B,D", [(3, 4096), (9, 1024), (5, 2240)])
def test_rows_without_the_shared_op_shift_table(ad, B, D):
    # B * D * 4 bytes above 32 KiB: the output pass reads scale / shift from
    # global memory instead of the per-CTA table
    assert B * D * 4 > 32 * 1024
    N = 24
    x = synth.normal_bits(D + 31, B * N * D, 0, 1).reshape(B, N, D)
    table = synth.normal_bits(D + 32, B * 2 * D, 0, 0.1).reshape(B, 2, D)
    got, ref = run_both(ad, x, B, N, D, (N * D, D, 1), table, D, 0, 2 * D, 1e-6, expect="rows")
    assert_bits_equal(got, ref, what=f"rows without table B={B} D={D}")


def test_rows_many_rows_per_warp(ad):
    # far more rows than resident warps: every warp handles many rows
    B, N, D = 1, 20000, 512
    x = synth.normal_bits(23, B * N * D, 0, 1).reshape(B, N, D)
    table = synth.normal_bits(24, 2 * D, 0, 0.1).reshape(1, 2, D)
    got, ref = run_both(ad, x, B, N, D, (N * D, D, 1), table, D, 0, 2 * D, 1e-6, expect="rows")
    assert_bits_equal(got, ref, what="many rows")
