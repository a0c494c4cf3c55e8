"""The torch layer's checks in front of the C ABI (which takes raw pointers
and cannot see where they point): CUDA tensors on the current device, one
storage dtype for the operands, and outputs that are contiguous, of the right
dtype and exactly as large as what the kernel writes.  Checked on the host
with stand-in tensors; host tensors are rejected before any CUDA call."""
import types

import pytest
import torch


@pytest.fixture(scope="module")
def ad():
    import __graft_entry__
    __graft_entry__.build()
    import adaln_modulate_gb300
    return adaln_modulate_gb300


class Fake:
    """Just the attributes the guard reads."""

    def __init__(self, dtype=torch.bfloat16, numel=8, device=0, cuda=True, contiguous=True):
        self.dtype, self._numel, self._device, self.is_cuda, self._contig = dtype, numel, device, cuda, contiguous

    def get_device(self):
        return self._device

    def numel(self):
        return self._numel

    def is_contiguous(self):
        return self._contig


@pytest.fixture
def guard(ad, monkeypatch):
    fake_torch = types.SimpleNamespace(cuda=types.SimpleNamespace(current_device=lambda: 0))
    monkeypatch.setattr(ad, "_torch", lambda: fake_torch)
    return ad._guard


def test_valid_calls_pass(guard):
    x = Fake()
    guard("op", x, (Fake(), None, Fake()), ((Fake(numel=8), 8, (torch.bfloat16,)), (None, 8, (torch.bfloat16,))))
    guard("op", x, others=(Fake(dtype=torch.float32),))
    guard("op", x, outs=((Fake(dtype=torch.uint8), 8, (torch.uint8, torch.float8_e4m3fn)),))


@pytest.mark.parametrize("bad", [Fake(cuda=False), Fake(device=1)])
def test_tensors_off_the_current_device(guard, bad):
    with pytest.raises(ValueError):
        guard("op", Fake(), (bad,))
    with pytest.raises(ValueError):
        guard("op", Fake(), others=(bad,))
    with pytest.raises(ValueError):
        guard("op", bad)


def test_operand_dtype_must_match(guard):
    with pytest.raises(TypeError):
        guard("op", Fake(), (Fake(dtype=torch.float16),))
    guard("op", Fake(), others=(Fake(dtype=torch.float16),))   # no dtype rule for these


@pytest.mark.parametrize("out", [Fake(numel=7), Fake(numel=9), Fake(contiguous=False), Fake(dtype=torch.float16)])
def test_bad_outputs(guard, out):
    with pytest.raises(ValueError):
        guard("op", Fake(), outs=((out, 8, (torch.bfloat16,)),))


def test_host_tensors_are_rejected_before_any_cuda_call(ad):
    x = torch.zeros((1, 4, 8), dtype=torch.bfloat16)
    rows = torch.zeros((1, 8), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ad.ln_modulate(x, rows, rows, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ad.rmsnorm_scale_shift(x, rows, rows, 1e-6)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ad.residual_gate_add(x, rows, x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ad.bias_gelu_tanh(x.view(4, 8), rows.view(8))
