"""The same-byte copy the measurements use as their yardstick
(adaln_copy_reference), through the C ABI: byte-exact for sizes with and
without a tail below 32 bytes, with and without the PDL flag, and its
argument checks."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [1, 31, 32, 33, 4096, 8192 + 17, (1 << 20) + 5, 9_184_000, 21_239_810])
@pytest.mark.parametrize("flags", [0, 1])
def test_copy_is_byte_exact(nbytes, flags):
    import adaln_modulate_gb300 as ad
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    src = torch.randint(0, 256, (nbytes + 64,), dtype=torch.uint8, device="cuda", generator=g)
    dst = torch.full((nbytes + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    st = ad.capi.adaln_copy_reference(dst.data_ptr(), src.data_ptr(), nbytes, flags,
                                      torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0
    assert torch.equal(dst[:nbytes], src[:nbytes])
    assert bool((dst[nbytes:] == 0xA5).all())       # nothing written past the end


def test_copy_argument_checks():
    import adaln_modulate_gb300 as ad
    f = ad.capi.adaln_copy_reference
    a = torch.empty(1 << 12, dtype=torch.uint8, device="cuda")
    b = torch.empty(1 << 12, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert f(None, b.data_ptr(), 64, 0, s) == 1                      # null
    assert f(a.data_ptr(), b.data_ptr(), 0, 0, s) == 3               # empty
    assert f(a.data_ptr() + 16, b.data_ptr(), 64, 0, s) == 4         # not 32-byte aligned
    assert f(a.data_ptr(), b.data_ptr(), 64, 2, s) == 6              # unknown flag
    assert f(a.data_ptr() + 32, a.data_ptr(), 64, 0, s) == 7         # overlap
