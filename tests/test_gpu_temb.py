"""GPU parity of adaln_temb_table_slices with the oracle, bit for bit, through
the C ABI: every dtype pair, the 8-wide and the scalar kernels, one row per
sample, one chunk, and a Wan-sized call checked on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import dev_tensor

pytestmark = pytest.mark.gpu

TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}


@pytest.fixture(scope="module")
def ad():
    import adaln_modulate_gb300
    assert torch.cuda.is_available()
    return adaln_modulate_gb300


def draw(seed, n, std, dt):
    if dt == "fp32":
        return (np.random.default_rng(seed).standard_normal(n) * std).astype(np.float32)
    return synth.normal_bits(seed, n, 0, std, dt)


def dev(a, dt):
    if dt == "fp32":
        return torch.from_numpy(np.ascontiguousarray(a)).cuda()
    return dev_tensor(a, dt)


def case(ad, B, S, K, D, table_dt="fp32", temb_dt="bf16", seed=0, out_offset=0):
    table = draw(seed, K * D, 0.05, table_dt).reshape(K, D)
    temb = draw(seed + 1, B * S * K * D, 1.0, temb_dt).reshape(B, S, K, D)
    out = None
    if out_offset:
        buf = torch.empty(K * B * S * D + out_offset, dtype=torch.float32, device="cuda")
        out = buf[out_offset:].view(K, B, S, D)
    slices = ad.temb_table_slices(dev(table, table_dt), dev(temb, temb_dt), out=out)
    torch.cuda.synchronize()
    ref = oracle.temb_table_slices(table, table_dt, temb, temb_dt, B, S, K, D)
    assert len(slices) == K
    for k, sl in enumerate(slices):
        assert sl.is_contiguous() and tuple(sl.shape) == (B, S, D)
        got = sl.cpu().numpy().view(np.uint32)
        exp = ref[k].view(np.uint32)
        bad = got != exp
        assert not bad.any(), f"slice {k}: {int(bad.sum())} mismatches ({table_dt}+{temb_dt}, D={D})"


@pytest.mark.parametrize("table_dt,temb_dt", [("fp32", "bf16"), ("bf16", "bf16"), ("fp32", "fp32"),
                                              ("fp16", "fp16"), ("bf16", "fp32"), ("fp32", "fp16")])
def test_dtype_pairs(ad, table_dt, temb_dt):
    case(ad, 2, 37, 6, 1536, table_dt, temb_dt, seed=len(table_dt + temb_dt))


@pytest.mark.parametrize("D", [1, 3, 12, 100, 1030])
def test_scalar_kernel_shapes(ad, D):
    case(ad, 2, 9, 6, D, seed=D)


def test_unaligned_output_takes_the_scalar_kernel(ad):
    case(ad, 1, 20, 6, 512, seed=5, out_offset=4)   # 16-byte, not 32-byte aligned


def test_one_row_per_sample_and_one_chunk(ad):
    case(ad, 3, 1, 6, 3072, seed=6)
    case(ad, 2, 50, 1, 256, seed=7)


def test_wan_sized_sampled_tokens(ad):
    # (1, 32760, 6, 3072) bf16 temb, binary32 table: tokens sampled for the oracle
    B, S, K, D = 1, 32760, 6, 3072
    table = draw(8, K * D, 0.05, "fp32").reshape(K, D)
    temb = draw(9, B * S * K * D, 1.0, "bf16").reshape(B, S, K, D)
    slices = ad.temb_table_slices(dev(table, "fp32"), dev(temb, "bf16"))
    torch.cuda.synchronize()
    sel = np.arange(0, S, 97)
    ref = oracle.temb_table_slices(table, "fp32", np.ascontiguousarray(temb[:, sel]), "bf16", B, sel.size, K, D)
    for k in range(K):
        got = slices[k][:, torch.from_numpy(sel).cuda()].cpu().numpy().view(np.uint32)
        assert np.array_equal(got, ref[k].view(np.uint32)), k
