"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds no arithmetic of the fused chains: it only draws random
16-bit storage values.  Both sides receive the same bytes from here and
nothing else in common.

The generator itself is ``synth.c`` (SplitMix64 counters + Box-Muller, see
that file), compiled on first use with gcc into ``synth/_build`` and run on
all host cores.  Element ``i`` of stream ``seed`` depends on ``(seed, i)``
only, so any slice can be drawn on its own (``first=``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple

import numpy as np

DTYPES = ("bf16", "fp16")
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile ``synth.c`` into ``synth/_build/libsynth.so`` (if stale)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-shared", "-fPIC", "-pthread", _SRC,
                    "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.synth_normal16.restype = ctypes.c_int
            lib.synth_normal16.argtypes = [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_uint64,
                                           ctypes.c_uint64, ctypes.c_double, ctypes.c_double,
                                           ctypes.c_int, ctypes.c_int]
            _lib = lib
    return _lib


def normal_bits(seed: int, n: int, mean: float = 0.0, std: float = 1.0,
                dtype: str = "bf16", first: int = 0,
                threads: Optional[int] = None) -> np.ndarray:
    """Elements ``[first, first+n)`` of stream ``seed`` drawn from N(mean, std)
    (``std`` is a standard deviation), as 16-bit storage patterns (uint16)."""
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().synth_normal16(out.ctypes.data, n, first, seed & 0xFFFFFFFFFFFFFFFF,
                               float(mean), float(std), DTYPES.index(dtype),
                               threads or (os.cpu_count() or 1))
    return out


# --------------------------------------------------------------------------
# Workload recipes.  Shapes, distributions and seeds of the five workloads
# the pages describe (Sana, GLM-Image, Wan2.2 and a tiny case).
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class TensorSpec:
    shape: Tuple[int, ...]
    mean: float
    std: float
    seed: int

    def draw(self, dtype: str = "bf16") -> np.ndarray:
        n = int(np.prod(self.shape)) if self.shape else 1
        return normal_bits(self.seed, n, self.mean, self.std, dtype).reshape(self.shape)


@dataclass(frozen=True)
class Workload:
    name: str
    op: str
    tensors: Dict[str, TensorSpec]
    params: Dict[str, object] = field(default_factory=dict)


# One seed per tensor role, so that no two tensors of a workload share a
# stream: 0 x (and q), 1 scale / adaLN table, 2 shift, 3-6 qk weights and
# biases, 7 GELU bias, 8 k, 9 y, 10 gate.
SEEDS = {"x": 0, "scale": 1, "table": 1, "shift": 2, "wq": 3, "bq": 4, "wk": 5,
         "bk": 6, "bias": 7, "k": 8, "y": 9, "gate": 10}


def ln_tiny() -> Workload:
    return Workload("ln_modulate tiny (1,64,512)", "ln_modulate", {
        "x": TensorSpec((1, 64, 512), 0.0, 1.0, SEEDS["x"]),
        "scale": TensorSpec((1, 1, 512), 0.0, 0.1, SEEDS["scale"]),
        "shift": TensorSpec((1, 1, 512), 0.0, 0.1, SEEDS["shift"]),
    }, {"eps": 1e-6})


def ln_sana(nmod: int = 6, scale_chunk: int = 1, shift_chunk: int = 0,
            transposed: bool = True, B: int = 2, N: int = 1024, D: int = 2240) -> Workload:
    """Sana block: x is the (B, N, D) view of a contiguous (B, D, N) tensor."""
    base = (B, D, N) if transposed else (B, N, D)
    return Workload(f"ln_modulate Sana ({B},{N},{D}) nmod={nmod}"
                    + (" transposed" if transposed else ""), "ln_modulate", {
        "x": TensorSpec(base, 0.0, 1.0, SEEDS["x"]),
        "table": TensorSpec((B, nmod, D), 0.0, 0.1, SEEDS["table"]),
    }, {"eps": 1e-6, "nmod": nmod, "scale_chunk": scale_chunk,
        "shift_chunk": shift_chunk, "transposed": transposed, "B": B, "N": N, "D": D})


def ln_glm() -> Workload:
    return Workload("ln_modulate GLM-Image (1,4096,4096)", "ln_modulate", {
        "x": TensorSpec((1, 4096, 4096), 0.0, 1.0, SEEDS["x"]),
        "scale": TensorSpec((1, 1, 4096), 0.0, 0.1, SEEDS["scale"]),
        "shift": TensorSpec((1, 1, 4096), 0.0, 0.1, SEEDS["shift"]),
    }, {"eps": 1e-5})


def gate_add_glm() -> Workload:
    return Workload("residual_gate_add GLM-Image (1,4096,4096)", "residual_gate_add", {
        "x": TensorSpec((1, 4096, 4096), 0.0, 1.0, SEEDS["x"]),
        "y": TensorSpec((1, 4096, 4096), 0.0, 1.0, SEEDS["y"]),
        "gate": TensorSpec((1, 1, 4096), 0.0, 0.1, SEEDS["gate"]),
    })


def qk_glm() -> Workload:
    return Workload("qk_head_layernorm GLM-Image (1,4360,32,128)", "qk_head_layernorm", {
        "q": TensorSpec((1, 4360, 32, 128), 0.0, 2.0, SEEDS["x"]),
        "k": TensorSpec((1, 4360, 32, 128), 0.0, 2.0, SEEDS["k"]),
        "wq": TensorSpec((128,), 1.0, 0.05, SEEDS["wq"]),
        "bq": TensorSpec((128,), 0.0, 0.05, SEEDS["bq"]),
        "wk": TensorSpec((128,), 1.0, 0.05, SEEDS["wk"]),
        "bk": TensorSpec((128,), 0.0, 0.05, SEEDS["bk"]),
    }, {"eps": 1e-6})


def gelu_wan(dtype: str = "bf16") -> Workload:
    return Workload(f"bias_gelu_tanh Wan2.2 (1,32760,13824) {dtype}", "bias_gelu_tanh", {
        "x": TensorSpec((32760, 13824), 0.0, 1.0, SEEDS["x"]),
        "bias": TensorSpec((13824,), 0.0, 0.02, SEEDS["bias"]),
    }, {"dtype": dtype})


def rms_rows(N: int = 4096, D: int = 4096) -> Workload:
    """RMSNorm + modulate with one scale / shift row per sample, the GLM
    LayerNorm's shape."""
    return Workload(f"rmsnorm_scale_shift (1,{N},{D}) per-sample rows", "rmsnorm_scale_shift", {
        "x": TensorSpec((1, N, D), 0.0, 1.0, SEEDS["x"]),
        "scale": TensorSpec((1, 1, D), 0.0, 0.1, SEEDS["scale"]),
        "shift": TensorSpec((1, 1, D), 0.0, 0.1, SEEDS["shift"]),
    }, {"eps": 1e-6})


def rms_tokens(N: int = 4096, D: int = 4096) -> Workload:
    """RMSNorm + modulate with per-token scale / shift: chunks 1 and 0 of a
    (1, N, 6, D) modulation table (the strided [B, S, 6D] chunk views)."""
    return Workload(f"rmsnorm_scale_shift (1,{N},{D}) per-token rows of a (1,{N},6,{D}) table",
                    "rmsnorm_scale_shift", {
                        "x": TensorSpec((1, N, D), 0.0, 1.0, SEEDS["x"]),
                        "table": TensorSpec((1, N, 6, D), 0.0, 0.1, SEEDS["table"]),
                    }, {"eps": 1e-6})


def gate_rms_tokens(N: int = 4096, D: int = 4096) -> Workload:
    """r = x + gate * y with a per-token [1, N, 1] gate, then RMSNorm(r) *
    (1 + scale) + shift with per-token rows of a (1, N, 6, D) table."""
    return Workload(f"norm_scale_shift rms (1,{N},{D}) per-token gate [1,{N},1] and rows",
                    "norm_scale_shift", {
                        "x": TensorSpec((1, N, D), 0.0, 1.0, SEEDS["x"]),
                        "y": TensorSpec((1, N, D), 0.0, 1.0, SEEDS["y"]),
                        "gate": TensorSpec((1, N, 1), 0.0, 0.5, SEEDS["gate"]),
                        "table": TensorSpec((1, N, 6, D), 0.0, 0.1, SEEDS["table"]),
                    }, {"eps": 1e-6})


def qk_rms(N: int = 4096, H: int = 30) -> Workload:
    """Per-head QK RMSNorm with weights, H heads of 128 over N tokens."""
    return Workload(f"qk_rmsnorm (1,{N},{H},128)", "qk_rmsnorm", {
        "q": TensorSpec((1, N, H, 128), 0.0, 2.0, SEEDS["x"]),
        "k": TensorSpec((1, N, H, 128), 0.0, 2.0, SEEDS["k"]),
        "wq": TensorSpec((128,), 1.0, 0.05, SEEDS["wq"]),
        "wk": TensorSpec((128,), 1.0, 0.05, SEEDS["wk"]),
    }, {"eps": 1e-6})


def temb_slices(S: int = 32760, K: int = 6, D: int = 3072) -> Workload:
    """A per-token modulation input: temb (1, S, K, D) bf16 and a binary32
    (K, D) table, the shape of the Wan FFN workload's tokens at width 3072."""
    return Workload(f"temb_table_slices (1,{S},{K},{D}) bf16 temb, binary32 table", "temb_table_slices", {
        "temb": TensorSpec((1, S, K, D), 0.0, 1.0, SEEDS["x"]),
        "table": TensorSpec((K, D), 0.0, 0.05, SEEDS["table"]),
    })


def ln_fp8_flux(N: int = 4608, D: int = 3072) -> Workload:
    """LayerNorm + modulate into static FP8 at a FLUX-like width: 4096 image
    and 512 text tokens of 3072 channels; static scale 0.03 (outputs span
    the e4m3 range and a few saturate)."""
    return Workload(f"ln_modulate_fp8 (1,{N},{D}) static e4m3 output", "ln_modulate_fp8", {
        "x": TensorSpec((1, N, D), 0.0, 1.0, SEEDS["x"]),
        "scale": TensorSpec((1, 1, D), 0.0, 0.1, SEEDS["scale"]),
        "shift": TensorSpec((1, 1, D), 0.0, 0.1, SEEDS["shift"]),
    }, {"eps": 1e-6, "qscale": 0.03})


def ln_wan(N: int = 32760, D: int = 5120) -> Workload:
    """LayerNorm + modulate on 5120-wide rows (the Wan FFN workload's
    tokens at the model width), one scale / shift row per sample."""
    return Workload(f"ln_modulate (1,{N},{D}) per-sample rows", "ln_modulate", {
        "x": TensorSpec((1, N, D), 0.0, 1.0, SEEDS["x"]),
        "scale": TensorSpec((1, 1, D), 0.0, 0.1, SEEDS["scale"]),
        "shift": TensorSpec((1, 1, D), 0.0, 0.1, SEEDS["shift"]),
    }, {"eps": 1e-6})


def all_workloads() -> List[Workload]:
    return [ln_tiny(), ln_sana(), ln_glm(), gate_add_glm(), qk_glm(), gelu_wan("bf16"),
            gelu_wan("fp16"), rms_rows(), rms_tokens(), gate_rms_tokens(), qk_rms(), temb_slices(),
            ln_fp8_flux(), ln_wan()]
