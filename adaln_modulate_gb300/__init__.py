"""Python binding of ``libadaln_gb300.so`` (the C ABI in ``include/adaln.h``).

Argument marshalling only: every operation runs in the library's sm_103a
kernels.  There is no fallback: if the library is not built, importing this
package raises ``ImportError`` (build it with ``__graft_entry__.build()`` or
``python adaln_modulate_gb300/_build.py``).

Two layers:
  * ``capi``: the C functions under their C names (``capi.adaln_ln_modulate``
    and so on), taking raw integers (device pointers, sizes, a stream handle);
  * ``ln_modulate``, ``qk_head_layernorm``, ``residual_gate_add``,
    ``bias_gelu_tanh``, ``residual_gate_ln_modulate``, ``norm_scale_shift``,
    ``rmsnorm_scale_shift``, ``qk_rmsnorm``, ``temb_table_slices``,
    ``ln_modulate_fp8``: the same calls taking torch tensors (PyTorch only
    provides the device memory and the current stream).
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional

from . import _build

LIB_PATH = _build.LIB
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "adaln.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run __graft_entry__.build() (nvcc, sm_103a)")

_lib = ctypes.CDLL(LIB_PATH)

BF16, FP16 = 0, 1
FLAG_PDL = 1
NORM = {"layer": 0, "rms": 1}
STATUS = {0: "ADALN_OK", 1: "ADALN_E_NULL", 2: "ADALN_E_DTYPE", 3: "ADALN_E_SHAPE",
          4: "ADALN_E_ALIGN", 5: "ADALN_E_STRIDE", 6: "ADALN_E_VALUE", 7: "ADALN_E_OVERLAP",
          8: "ADALN_E_CUDA"}
VARIANTS = {0: "rows", 1: "tokens", 2: "generic", 3: "tokens_tma"}

_P, _I, _F, _U, _INT = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_uint32, ctypes.c_int
_SIGS = {
    "adaln_status_str": ([_INT], ctypes.c_char_p),
    "adaln_last_cuda_error": ([], ctypes.c_char_p),
    "adaln_version": ([], _INT),
    "adaln_init": ([_INT], _INT),
    "adaln_shutdown": ([], _INT),
    "adaln_ln_modulate": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U, _P], _INT),
    "adaln_can_ln_modulate": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U], _INT),
    "adaln_ln_modulate_variant": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U],
                                  _INT),
    "adaln_qk_head_layernorm": ([_P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P, _F, _INT, _U, _P], _INT),
    "adaln_can_qk_head_layernorm": ([_P, _P, _I, _P, _P, _I, _I, _P, _P, _P, _P, _F, _INT, _U],
                                    _INT),
    "adaln_residual_gate_add": ([_P, _P, _P, _I, _P, _I, _I, _I, _INT, _U, _P], _INT),
    "adaln_can_residual_gate_add": ([_P, _P, _P, _I, _P, _I, _I, _I, _INT, _U], _INT),
    "adaln_bias_gelu_tanh": ([_P, _P, _P, _I, _I, _INT, _U, _P], _INT),
    "adaln_can_bias_gelu_tanh": ([_P, _P, _P, _I, _I, _INT, _U], _INT),
    "adaln_bias_gelu_tanh_noalloc": ([_P, _P, _P, _I, _I, _INT, _U, _P], _INT),
    "adaln_copy_reference": ([_P, _P, _I, _U, _P], _INT),
    "adaln_tma_wait_timeouts": ([_P], _INT),
    "adaln_residual_gate_ln_modulate": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U, _P],
                                        _INT),
    "adaln_can_residual_gate_ln_modulate": ([_P, _P, _P, _P, _I, _P, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U],
                                            _INT),
    "adaln_norm_scale_shift": ([_INT, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _I, _P, _P, _I, _I, _P, _I,
                                _I, _F, _INT, _U, _P], _INT),
    "adaln_can_norm_scale_shift": ([_INT, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _I, _P, _P, _I, _I, _P,
                                    _I, _I, _F, _INT, _U], _INT),
    "adaln_norm_scale_shift_variant": ([_INT, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _I, _P, _P, _I, _I,
                                        _P, _I, _I, _F, _INT, _U], _INT),
    "adaln_rmsnorm_scale_shift": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _P, _I, _I, _F, _INT, _U, _P], _INT),
    "adaln_can_rmsnorm_scale_shift": ([_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _P, _I, _I, _F, _INT, _U], _INT),
    "adaln_qk_rmsnorm": ([_P, _P, _I, _P, _P, _I, _I, _P, _P, _F, _INT, _U, _P], _INT),
    "adaln_can_qk_rmsnorm": ([_P, _P, _I, _P, _P, _I, _I, _P, _P, _F, _INT, _U], _INT),
    "adaln_temb_table_slices": ([_P, _I, _P, _INT, _P, _INT, _I, _I, _I, _I, _U, _P], _INT),
    "adaln_ln_modulate_fp8": ([_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U, _P], _INT),
    "adaln_can_ln_modulate_fp8": ([_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U], _INT),
    "adaln_ln_modulate_fp8_variant": ([_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT, _U], _INT),
    "adaln_can_temb_table_slices": ([_P, _I, _P, _INT, _P, _INT, _I, _I, _I, _I, _U], _INT),
}


class _CApi:
    """The C entry points under their C names."""

    def __init__(self, lib):
        for name, (args, res) in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
            setattr(self, name, fn)


capi = _CApi(_lib)


def header_functions() -> list:
    """Names of every function declared in include/adaln.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(adaln_\w+)\s*\(", text)))


class AdalnError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {STATUS.get(status, status)}"
        if status == 8:
            msg += f" ({capi.adaln_last_cuda_error().decode()})"
        super().__init__(msg)
        self.status = status


def _check(status: int, where: str) -> None:
    if status != 0:
        raise AdalnError(status, where)


# ------------------------------------------------------------------ torch

def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float16:
        return FP16
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 / fp16 only)")


def _stream(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _guard(where: str, ref, inputs=(), outs=(), others=()) -> None:
    """The C ABI takes raw pointers and cannot see where they point, so the
    torch layer checks what it can: every tensor is a CUDA tensor on the
    current device (``others``: no dtype rule), every entry of ``inputs``
    has ``ref``'s dtype, and every output given as (tensor, element count,
    dtypes) is contiguous with that many elements of one of those dtypes
    (a smaller buffer would be written past its end)."""
    tensors = [t for t in (ref, *inputs, *others, *(o[0] for o in outs)) if t is not None]
    if not all(t.is_cuda for t in tensors):
        raise ValueError(f"{where}: every tensor must be a CUDA tensor")
    dev = _torch().cuda.current_device()
    if any(t.get_device() != dev for t in tensors):
        raise ValueError(f"{where}: every tensor must be on the current CUDA device (cuda:{dev})")
    for t in inputs:
        if t is not None and t.dtype != ref.dtype:
            raise TypeError(f"{where}: a {t.dtype} operand with a {ref.dtype} input")
    for t, numel, dtypes in outs:
        if t is not None and (t.dtype not in dtypes or t.numel() != numel or not t.is_contiguous()):
            raise ValueError(f"{where}: the output must be a contiguous tensor of {numel} elements of {dtypes}")


def _rows_view(t, D: int, name: str):
    """(pointer, batch stride) of a (B, D) / (B, 1, D) row tensor."""
    if t.dim() == 3:
        if t.shape[1] != 1:
            raise ValueError(f"{name} must be (B, 1, D)")
        t = t[:, 0]
    if t.dim() == 1:
        t = t.unsqueeze(0)
    if t.dim() != 2 or t.shape[-1] != D or (D > 1 and t.stride(-1) != 1):
        raise ValueError(f"{name} must be (B, D) rows contiguous over D")
    return t.data_ptr(), (t.stride(0) if t.shape[0] > 1 else 0)


def ln_modulate(x, scale, shift, eps: float, out=None, flags: int = 0, stream=None):
    """``LN(x) * (1 + scale) + shift`` for x (B, N, D) of any strides;
    scale / shift (B, 1, D) or (B, D) with contiguous rows.  Returns the
    contiguous (B, N, D) output."""
    torch = _torch()
    B, N, D = x.shape
    _guard("ln_modulate", x, (scale, shift), ((out, B * N * D, (x.dtype,)),))
    if out is None:
        out = torch.empty((B, N, D), dtype=x.dtype, device=x.device)
    sp, ssb = _rows_view(scale, D, "scale")
    hp, hsb = _rows_view(shift, D, "shift")
    if scale.shape[0] not in (1, B) or shift.shape[0] not in (1, B):
        raise ValueError("scale / shift batch must be 1 or B")
    if scale.shape[0] == 1:
        ssb = 0
    if shift.shape[0] == 1:
        hsb = 0
    st = capi.adaln_ln_modulate(out.data_ptr(), x.data_ptr(), B, N, D, *x.stride(), sp, ssb, hp,
                                hsb, float(eps), _dtype_code(x), flags, _stream(stream))
    _check(st, "adaln_ln_modulate")
    return out


def _fp8_args(x, scale, shift, qscale):
    B, N, D = x.shape
    rows = []
    for t, name in ((scale, "scale"), (shift, "shift")):
        p, sb = _rows_view(t, D, name)
        if t.shape[0] not in (1, B):
            raise ValueError(f"{name} batch must be 1 or B")
        rows.append((p, 0 if t.shape[0] == 1 else sb))
    if qscale.numel() != 1 or qscale.dtype != _torch().float32:
        raise ValueError("qscale must be one float32 value on the device")
    return B, N, D, rows


def ln_modulate_fp8(x, scale, shift, eps: float, qscale, out=None, flags: int = 0, stream=None):
    """``e4m3((LN(x) * (1 + scale) + shift) / qscale)`` (static FP8) for x
    (B, N, D) of any strides; scale / shift as ln_modulate; qscale a float32
    device tensor of one element.  Returns a (B, N, D) torch.float8_e4m3fn
    tensor (or writes ``out``, uint8 or float8_e4m3fn)."""
    torch = _torch()
    B, N, D, ((sp, ssb), (hp, hsb)) = _fp8_args(x, scale, shift, qscale)
    _guard("ln_modulate_fp8", x, (scale, shift), ((out, B * N * D, (torch.uint8, torch.float8_e4m3fn)),),
           others=(qscale,))
    if out is None:
        out = torch.empty((B, N, D), dtype=torch.float8_e4m3fn, device=x.device)
    st = capi.adaln_ln_modulate_fp8(out.data_ptr(), qscale.data_ptr(), x.data_ptr(), B, N, D, *x.stride(), sp, ssb,
                                    hp, hsb, float(eps), _dtype_code(x), flags, _stream(stream))
    _check(st, "adaln_ln_modulate_fp8")
    return out


def ln_modulate_fp8_variant(x, scale, shift, eps: float, qscale) -> str:
    """Which kernel ln_modulate_fp8 takes for these tensors (no CUDA work)."""
    B, N, D, ((sp, ssb), (hp, hsb)) = _fp8_args(x, scale, shift, qscale)
    v = capi.adaln_ln_modulate_fp8_variant(1 << 40, qscale.data_ptr(), x.data_ptr(), B, N, D, *x.stride(), sp, ssb,
                                           hp, hsb, float(eps), _dtype_code(x), 0)
    if v < 0:
        raise AdalnError(-v, "adaln_ln_modulate_fp8_variant")
    return VARIANTS[v]


def tma_wait_timeouts() -> int:
    """Bounded TMA waits that gave up on the current device (diagnostic; 0)."""
    n = ctypes.c_uint32(0)
    _check(capi.adaln_tma_wait_timeouts(ctypes.byref(n)), "adaln_tma_wait_timeouts")
    return n.value


def ln_modulate_variant(x, scale, shift, eps: float, out=None) -> str:
    """Which kernel ln_modulate takes for these tensors (no CUDA work)."""
    B, N, D = x.shape
    sp, ssb = _rows_view(scale, D, "scale")
    hp, hsb = _rows_view(shift, D, "shift")
    optr = out.data_ptr() if out is not None else 1 << 40
    v = capi.adaln_ln_modulate_variant(optr, x.data_ptr(), B, N, D, *x.stride(), sp, ssb, hp, hsb,
                                       float(eps), _dtype_code(x), 0)
    if v < 0:
        raise AdalnError(-v, "adaln_ln_modulate_variant")
    return VARIANTS[v]


def qk_head_layernorm(q, k, wq, bq, wk, bk, eps: float, q_out=None, k_out=None, flags: int = 0,
                      stream=None):
    """Per-head LayerNorm with affine of q and k (any leading shape, last
    dim Dh, contiguous) in one launch.  Pass ``q_out=q`` for in place."""
    torch = _torch()
    Dh = q.shape[-1] if q is not None else k.shape[-1]
    rq = q.numel() // Dh if q is not None else 0
    rk = k.numel() // Dh if k is not None else 0
    for t in (q, k):
        if t is not None and not t.is_contiguous():
            raise ValueError("q / k must be contiguous")
    ref = q if q is not None else k
    _guard("qk_head_layernorm", ref, (q, k, wq, bq, wk, bk),
           ((q_out, rq * Dh, (ref.dtype,)), (k_out, rk * Dh, (ref.dtype,))))
    if q is not None and q_out is None:
        q_out = torch.empty_like(q)
    if k is not None and k_out is None:
        k_out = torch.empty_like(k)
    ptr = lambda t: t.data_ptr() if t is not None else None
    st = capi.adaln_qk_head_layernorm(ptr(q_out), ptr(q), rq, ptr(k_out), ptr(k), rk, Dh, ptr(wq),
                                      ptr(bq), ptr(wk), ptr(bk), float(eps), _dtype_code(ref), flags,
                                      _stream(stream))
    _check(st, "adaln_qk_head_layernorm")
    return q_out, k_out


def residual_gate_add(x, gate, y, out=None, flags: int = 0, stream=None):
    """``x + gate * y`` for contiguous x, y (B, N, D) and gate (B, 1, D) / (B, D)."""
    torch = _torch()
    B, N, D = x.shape
    if not (x.is_contiguous() and y.is_contiguous()) or y.shape != x.shape:
        raise ValueError("x and y must be contiguous (B, N, D)")
    _guard("residual_gate_add", x, (gate, y), ((out, B * N * D, (x.dtype,)),))
    if out is None:
        out = torch.empty_like(x)
    gp, gsb = _rows_view(gate, D, "gate")
    if gate.shape[0] == 1:
        gsb = 0
    st = capi.adaln_residual_gate_add(out.data_ptr(), x.data_ptr(), gp, gsb, y.data_ptr(), B, N, D,
                                      _dtype_code(x), flags, _stream(stream))
    _check(st, "adaln_residual_gate_add")
    return out


def residual_gate_ln_modulate(x, gate, y, scale, shift, eps: float, r_out=None, out=None, flags: int = 0,
                              stream=None):
    """``r = x + gate * y`` and ``LN(r) * (1 + scale) + shift`` in one pass for
    contiguous x, y (B, N, D); gate / scale / shift (B, 1, D) or (B, D) rows.
    Pass ``r_out=x`` for an in-place residual update.  Returns (r, out)."""
    torch = _torch()
    B, N, D = x.shape
    if not (x.is_contiguous() and y.is_contiguous()) or y.shape != x.shape:
        raise ValueError("x and y must be contiguous (B, N, D)")
    _guard("residual_gate_ln_modulate", x, (gate, y, scale, shift),
           ((r_out, B * N * D, (x.dtype,)), (out, B * N * D, (x.dtype,))))
    if r_out is None:
        r_out = torch.empty_like(x)
    if out is None:
        out = torch.empty_like(x)
    rows = []
    for t, name in ((gate, "gate"), (scale, "scale"), (shift, "shift")):
        p, sb = _rows_view(t, D, name)
        if t.shape[0] not in (1, B):
            raise ValueError(f"{name} batch must be 1 or B")
        rows.append((p, 0 if t.shape[0] == 1 else sb))
    (gp, gsb), (sp, ssb), (hp, hsb) = rows
    st = capi.adaln_residual_gate_ln_modulate(r_out.data_ptr(), out.data_ptr(), x.data_ptr(), gp, gsb,
                                              y.data_ptr(), B, N, D, sp, ssb, hp, hsb, float(eps),
                                              _dtype_code(x), flags, _stream(stream))
    _check(st, "adaln_residual_gate_ln_modulate")
    return r_out, out


def _operand(t, B: int, N: int, D: int, name: str, scalar_ok: bool = False):
    """(pointer, s_b, s_n, s_d) of an operand broadcast to (B, N, D): (D,),
    (B, D) / (1, D) rows per sample, or a 3-d (B|1, N|1, D) view (per-token
    rows, e.g. a chunk of a (B, N, 6, D) table); with ``scalar_ok`` also
    (B|1, N|1, 1), one value per token.  Broadcast dimensions get stride 0."""
    if t.dim() == 1:
        t = t.view(1, 1, -1)
    elif t.dim() == 2:
        t = t.unsqueeze(1)
    if t.dim() != 3:
        raise ValueError(f"{name} must be (D,), (B, D) or (B|1, N|1, D)")
    b, n, d = t.shape
    if b not in (1, B) or n not in (1, N) or d not in ((1, D) if scalar_ok else (D,)):
        raise ValueError(f"{name} of shape {tuple(t.shape)} does not broadcast to ({B}, {N}, {D})")
    if d > 1 and t.stride(2) != 1:
        raise ValueError(f"{name} must be contiguous over D")
    return (t.data_ptr(), t.stride(0) if b > 1 else 0, t.stride(1) if n > 1 else 0,
            1 if d > 1 else 0)


def _norm_call(fn, norm, x, scale, shift, eps, gate, y, r_out, out, flags, stream, variant=False):
    torch = _torch()
    B, N, D = x.shape
    if not variant:
        _guard("norm_scale_shift", x, (scale, shift, gate, y),
               ((r_out if gate is not None else None, B * N * D, (x.dtype,)), (out, B * N * D, (x.dtype,))))
    sp, ssb, ssn, _ = _operand(scale, B, N, D, "scale")
    hp, hsb, hsn, _ = _operand(shift, B, N, D, "shift")
    if gate is not None:
        if y is None or tuple(y.shape) != (B, N, D) or not y.is_contiguous() or not x.is_contiguous():
            raise ValueError("with a gate, x and y must be contiguous (B, N, D)")
        gp, gsb, gsn, gsd = _operand(gate, B, N, D, "gate", scalar_ok=True)
        if r_out is None and not variant:
            r_out = torch.empty_like(x)
        yp = y.data_ptr()
    else:
        gp, gsb, gsn, gsd, yp = None, 0, 0, 1, None
    if out is None and not variant:
        out = torch.empty((B, N, D), dtype=x.dtype, device=x.device)
    ptr = lambda t, dflt=None: t.data_ptr() if t is not None else dflt
    args = [NORM[norm], ptr(r_out, 1 << 41 if gate is not None else None), ptr(out, 1 << 40), x.data_ptr(), B, N,
            D, *x.stride(), gp, gsb, gsn, gsd, yp, sp, ssb, ssn, hp, hsb, hsn, float(eps), _dtype_code(x), flags]
    if variant:
        return fn(*args)
    _check(fn(*args, _stream(stream)), "adaln_norm_scale_shift")
    return (r_out, out) if gate is not None else out


def norm_scale_shift(x, scale, shift, eps: float, norm: str = "layer", gate=None, y=None, r_out=None, out=None,
                     flags: int = 0, stream=None):
    """``norm(v) * (1 + scale) + shift`` with ``norm`` "layer" (LayerNorm) or
    "rms" (RMSNorm), both without affine, and v = x, or, with ``gate``,
    v = x + gate * y (stored in ``r_out``; pass ``r_out=x`` to update x in
    place).  x is (B, N, D) of any strides (contiguous with a gate); scale /
    shift are (D,), (B, D), (B, 1, D) rows per sample or (B, N, D) views per
    token; gate is a per-sample row, a per-token row, or (B, N, 1) one value
    per token.  Returns out, or (r, out) with a gate."""
    return _norm_call(capi.adaln_norm_scale_shift, norm, x, scale, shift, eps, gate, y, r_out, out, flags, stream)


def norm_scale_shift_variant(x, scale, shift, eps: float, norm: str = "layer", gate=None, y=None, r_out=None,
                             out=None) -> str:
    """Which kernel norm_scale_shift takes for these tensors (no CUDA work)."""
    v = _norm_call(capi.adaln_norm_scale_shift_variant, norm, x, scale, shift, eps, gate, y, r_out, out, 0, None,
                   variant=True)
    if v < 0:
        raise AdalnError(-v, "adaln_norm_scale_shift_variant")
    return VARIANTS[v]


def rmsnorm_scale_shift(x, scale, shift, eps: float, out=None, flags: int = 0, stream=None):
    """``RMSNorm(x) * (1 + scale) + shift`` (no affine): norm_scale_shift
    with ``norm="rms"`` and no gate, through adaln_rmsnorm_scale_shift."""
    torch = _torch()
    B, N, D = x.shape
    _guard("rmsnorm_scale_shift", x, (scale, shift), ((out, B * N * D, (x.dtype,)),))
    sp, ssb, ssn, _ = _operand(scale, B, N, D, "scale")
    hp, hsb, hsn, _ = _operand(shift, B, N, D, "shift")
    if out is None:
        out = torch.empty((B, N, D), dtype=x.dtype, device=x.device)
    st = capi.adaln_rmsnorm_scale_shift(out.data_ptr(), x.data_ptr(), B, N, D, *x.stride(), sp, ssb, ssn, hp, hsb,
                                        hsn, float(eps), _dtype_code(x), flags, _stream(stream))
    _check(st, "adaln_rmsnorm_scale_shift")
    return out


def qk_rmsnorm(q, k, wq, wk, eps: float, q_out=None, k_out=None, flags: int = 0, stream=None):
    """Per-head RMSNorm with a weight of q and k (any leading shape, last dim
    Dh, contiguous) in one launch.  Pass ``q_out=q`` for in place."""
    torch = _torch()
    Dh = q.shape[-1] if q is not None else k.shape[-1]
    rq = q.numel() // Dh if q is not None else 0
    rk = k.numel() // Dh if k is not None else 0
    for t in (q, k):
        if t is not None and not t.is_contiguous():
            raise ValueError("q / k must be contiguous")
    ref = q if q is not None else k
    _guard("qk_rmsnorm", ref, (q, k, wq, wk), ((q_out, rq * Dh, (ref.dtype,)), (k_out, rk * Dh, (ref.dtype,))))
    if q is not None and q_out is None:
        q_out = torch.empty_like(q)
    if k is not None and k_out is None:
        k_out = torch.empty_like(k)
    ptr = lambda t: t.data_ptr() if t is not None else None
    st = capi.adaln_qk_rmsnorm(ptr(q_out), ptr(q), rq, ptr(k_out), ptr(k), rk, Dh, ptr(wq), ptr(wk), float(eps),
                               _dtype_code(ref), flags, _stream(stream))
    _check(st, "adaln_qk_rmsnorm")
    return q_out, k_out


def _any_dtype_code(t) -> int:
    torch = _torch()
    return 2 if t.dtype == torch.float32 else _dtype_code(t)


def temb_table_slices(table, temb, out=None, flags: int = 0, stream=None):
    """``(table + temb.float()).chunk(K, dim=2)`` as K contiguous float32
    tensors (B, S, D), written in one pass.  table (K, D) or (1, K, D); temb
    (B, S, K, D) or (B, K, D) (one row per sample), both contiguous, bf16,
    fp16 or float32.  ``out`` may be a (K, B, S, D) float32 buffer.  Returns
    the list of the K slices (views of one buffer)."""
    torch = _torch()
    if temb.dim() == 3:
        temb = temb.unsqueeze(1)
    B, S, K, D = temb.shape
    table = table.reshape(-1, table.shape[-1])
    if tuple(table.shape) != (K, D) or not table.is_contiguous() or not temb.is_contiguous():
        raise ValueError("table (K, D) and temb (B, S, K, D) must be contiguous")
    _guard("temb_table_slices", temb, others=(table, out))
    if out is None:
        out = torch.empty((K, B, S, D), dtype=torch.float32, device=temb.device)
    if tuple(out.shape) != (K, B, S, D) or out.dtype != torch.float32 or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 (K, B, S, D) buffer")
    st = capi.adaln_temb_table_slices(out.data_ptr(), B * S * D, table.data_ptr(), _any_dtype_code(table),
                                      temb.data_ptr(), _any_dtype_code(temb), B, S, K, D, flags, _stream(stream))
    _check(st, "adaln_temb_table_slices")
    return list(out.unbind(0))


def bias_gelu_tanh(x, bias, out=None, flags: int = 0, stream=None):
    """``gelu_tanh(round(x + bias))`` for contiguous x (..., width), bias (width,)."""
    torch = _torch()
    width = x.shape[-1]
    if not x.is_contiguous() or bias.numel() != width or not bias.is_contiguous():
        raise ValueError("x contiguous (..., width), bias (width,)")
    _guard("bias_gelu_tanh", x, (bias,), ((out, x.numel(), (x.dtype,)),))
    if out is None:
        out = torch.empty_like(x)
    st = capi.adaln_bias_gelu_tanh(out.data_ptr(), x.data_ptr(), bias.data_ptr(),
                                   x.numel() // width, width, _dtype_code(x), flags, _stream(stream))
    _check(st, "adaln_bias_gelu_tanh")
    return out


def copy_reference(src, dst, nbytes: Optional[int] = None, flags: int = 0, stream=None):
    """Same-byte device copy (the measurement yardstick): the first nbytes
    (default: all) bytes of src into dst, both CUDA tensors on this device."""
    _guard("copy_reference", dst, others=(src,))
    if not src.is_contiguous() or not dst.is_contiguous():
        raise ValueError("copy_reference: src and dst must be contiguous")
    n = src.numel() * src.element_size() if nbytes is None else int(nbytes)
    if n > src.numel() * src.element_size() or n > dst.numel() * dst.element_size():
        raise ValueError("copy_reference: nbytes beyond a tensor")
    st = capi.adaln_copy_reference(dst.data_ptr(), src.data_ptr(), n, flags, _stream(stream))
    _check(st, "adaln_copy_reference")
    return dst


def init(device: Optional[int] = None) -> None:
    """Build the per-device GELU tables now (needed before graph capture)."""
    if device is None:
        device = _torch().cuda.current_device()
    _check(capi.adaln_init(int(device)), "adaln_init")
