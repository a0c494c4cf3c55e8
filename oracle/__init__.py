"""CPU oracle for the fused DiT chains -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference arms may import this package.  The CUDA library and its
Python binding never touch it; the two share no code.

The arithmetic lives in ``oracle.c`` (plain scalar C, IEEE binary32 with
explicit ``fmaf``, built with ``-ffp-contract=off``); this module only
compiles it with gcc and marshals numpy arrays.  Every array of storage
values is ``uint16`` (bf16 or fp16 bit patterns).  Each function cites the
passage it follows in ``oracle.c``.

Parity status of each function (what pins it, see ``tests/test_oracle_*``):
  ln_modulate        pinned: fp64 two-pass LayerNorm, exact-arithmetic
                     cases, modulate identities, bit-level symmetries
  qk_head_layernorm  pinned: fp64 two-pass LayerNorm with affine, exact cases
  residual_gate_add  pinned: single-rounding fp64 definition
  norm_scale_shift   pinned: LN mode equals ln_modulate / the gate-add + LN
                     composition; RMS mode: fp64 RMSNorm, exact rows,
                     sign-flip and power-of-two symmetries; per-token rows
                     and gates equal per-row calls of the pinned forms
  qk_rmsnorm         pinned: fp64 RMSNorm with weight, exact rows
  temb_table_slices  pinned: numpy's binary32 addition of the promoted
                     operands, slice by slice
  e4m3 / quant_e4m3  pinned: torch's float8_e4m3fn rounding of clamped
                     values (every bf16 and fp16 pattern, tie cases),
                     exhaustive decode round trip; ln_modulate_fp8 is the
                     pinned LN+modulate followed by the pinned quantiser
  bias_gelu_tanh     pinned: 100-bit evaluation of tanh-GELU on all inputs
  rsqrt_cr           pinned: 100-bit evaluation
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_DEFAULT_LIB = _LIB_PATH
CFLAGS = ["-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fno-builtin",
          "-Wall", "-shared", "-fPIC"]
_lib = None
_lock = threading.Lock()

DTYPE_CODE = {"bf16": 0, "fp16": 1}
ANY_DTYPE_CODE = {"bf16": 0, "fp16": 1, "fp32": 2}


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/_build/liboracle.so`` (if stale)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int


def _lib_handle():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build() if _LIB_PATH == _DEFAULT_LIB else _LIB_PATH)
            sig = {
                "oracle_ln_modulate": [_P, _P, _I, _I, _I, _I, _I, _I, _P, _I, _P, _I, _F, _INT,
                                       _I, _I, _P, _P],
                "oracle_qk_head_layernorm": [_P, _P, _I, _I, _P, _P, _F, _INT, _I, _I],
                "oracle_residual_gate_add": [_P, _P, _P, _I, _P, _I, _I, _I, _INT, _I, _I],
                "oracle_bias_gelu_tanh": [_P, _P, _P, _I, _I, _INT, _I, _I],
                "oracle_gelu_table": [_P, _INT],
                "oracle_row_stats": [_P, _I, _INT, _P, _P],
                "oracle_row_sumsq": [_P, _I, _INT, _P],
                "oracle_norm_scale_shift": [_P, _P, _INT, _P, _I, _I, _I, _I, _I, _I, _P, _I, _I, _I, _P,
                                            _P, _I, _I, _P, _I, _I, _F, _INT, _I, _I, _P, _P],
                "oracle_qk_rmsnorm": [_P, _P, _I, _I, _P, _F, _INT, _I, _I],
                "oracle_temb_table_slices": [_P, _I, _P, _INT, _P, _INT, _I, _I, _I, _I],
                "oracle_quant_e4m3": [_P, _P, _I, _F, _INT],
            }
            for name, args in sig.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = ctypes.c_int
            for name, args in {"oracle_f32_to_16": [_P, _P, _I, _INT],
                               "oracle_f32_to_e4m3_array": [_P, _P, _I],
                               "oracle_16_to_f32": [_P, _P, _I, _INT],
                               "oracle_rsqrt_cr_array": [_P, _P, _I]}.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = None
            lib.oracle_rsqrt_cr.argtypes = [_F]
            lib.oracle_rsqrt_cr.restype = _F
            _lib = lib
    return _lib


class loaded_from:
    """Context manager: route every call of this module to another build of
    the oracle (used by the test that plants mistakes in a copy of
    ``oracle.c`` and checks that the pins catch them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        self.saved = (_lib, dict(_tables))
        _lib = None
        _tables.clear()
        real = _LIB_PATH
        globals()["_LIB_PATH"] = self.path
        try:
            _lib_handle()
        finally:
            globals()["_LIB_PATH"] = real
        return self

    def __exit__(self, *exc):
        global _lib
        _lib, tables = self.saved
        _tables.clear()
        _tables.update(tables)
        return False



def _u16(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("storage arrays are uint16 bit patterns")
    return a


def _segments(rows: Optional[Sequence[int]], total: int) -> Tuple[np.ndarray, list]:
    """Sorted row indices and their maximal contiguous runs [(begin, end), ...]."""
    if rows is None:
        idx = np.arange(total, dtype=np.int64)
    else:
        idx = np.asarray(sorted(set(int(r) for r in rows)), dtype=np.int64)
        if idx.size and (idx[0] < 0 or idx[-1] >= total):
            raise IndexError("row index out of range")
    runs = []
    if idx.size:
        start = prev = int(idx[0])
        for r in idx[1:]:
            r = int(r)
            if r != prev + 1:
                runs.append((start, prev + 1))
                start = r
            prev = r
        runs.append((start, prev + 1))
    return idx, runs


def _split_runs(runs, threads: int):
    """Split runs into about `threads` pieces of similar size for a pool."""
    total = sum(e - b for b, e in runs)
    if threads <= 1 or total < 2 * threads:
        return runs
    step = max(1, total // (threads * 4))
    out = []
    for b, e in runs:
        while b < e:
            out.append((b, min(e, b + step)))
            b += step
    return out


def _run(pieces, fn, threads):
    if threads <= 1 or len(pieces) <= 1:
        for p in pieces:
            fn(p)
    else:
        with ThreadPoolExecutor(max_workers=threads) as pool:
            list(pool.map(fn, pieces))


# --------------------------------------------------------------------------
# the four chains
# --------------------------------------------------------------------------

def ln_modulate(x_base: np.ndarray, B: int, N: int, D: int, strides: Tuple[int, int, int],
                scale_base: np.ndarray, scale_offset: int, s_scale_b: int,
                shift_base: np.ndarray, shift_offset: int, s_shift_b: int,
                eps: float, dtype: str = "bf16", rows: Optional[Sequence[int]] = None,
                threads: int = 1, return_stats: bool = False):
    """LayerNorm (no affine) + adaLN modulate on rows ``r = b*N + n``.

    ``x_base`` is the flat storage buffer; element (b, n, d) sits at
    ``b*sxB + n*sxN + d*sxD``.  ``scale``/``shift`` row b starts at
    ``offset + b*s_b`` of their buffers.  Returns ``(row_ids, out)`` with
    ``out`` of shape ``(len(row_ids), D)``; with ``return_stats`` also the
    per-row binary32 mean and rstd.
    """
    lib = _lib_handle()
    xb, sb, hb = _u16(x_base).reshape(-1), _u16(scale_base).reshape(-1), _u16(shift_base).reshape(-1)
    idx, runs = _segments(rows, B * N)
    out = np.zeros((idx.size, D), dtype=np.uint16)
    mean = np.zeros(idx.size, dtype=np.float32)
    rstd = np.zeros(idx.size, dtype=np.float32)
    pos = {int(r): i for i, r in enumerate(idx)}
    sxB, sxN, sxD = strides
    pieces = _split_runs(runs, threads)

    def one(piece):
        b0, e0 = piece
        i0 = pos[b0]
        rc = lib.oracle_ln_modulate(out[i0:].ctypes.data, xb.ctypes.data, B, N, D, sxB, sxN, sxD,
                                    sb.ctypes.data + 2 * scale_offset, s_scale_b,
                                    hb.ctypes.data + 2 * shift_offset, s_shift_b, eps,
                                    DTYPE_CODE[dtype], b0, e0, mean[i0:].ctypes.data,
                                    rstd[i0:].ctypes.data)
        if rc:
            raise ValueError(f"oracle_ln_modulate rejected its arguments ({rc})")

    _run(pieces, one, threads)
    if return_stats:
        return idx, out, mean, rstd
    return idx, out


def qk_head_layernorm(x: np.ndarray, Dh: int, w: np.ndarray, b: np.ndarray, eps: float,
                      dtype: str = "bf16", rows: Optional[Sequence[int]] = None,
                      threads: int = 1):
    """Per-head LayerNorm with affine on a (rows, Dh) tensor; returns (row_ids, out)."""
    lib = _lib_handle()
    xf = _u16(x).reshape(-1)
    nrows = xf.size // Dh
    w, b = _u16(w).reshape(-1), _u16(b).reshape(-1)
    idx, runs = _segments(rows, nrows)
    out = np.zeros((idx.size, Dh), dtype=np.uint16)
    pos = {int(r): i for i, r in enumerate(idx)}

    def one(piece):
        b0, e0 = piece
        rc = lib.oracle_qk_head_layernorm(out[pos[b0]:].ctypes.data, xf.ctypes.data, nrows, Dh,
                                          w.ctypes.data, b.ctypes.data, eps, DTYPE_CODE[dtype],
                                          b0, e0)
        if rc:
            raise ValueError(f"oracle_qk_head_layernorm rejected its arguments ({rc})")

    _run(_split_runs(runs, threads), one, threads)
    return idx, out


def residual_gate_add(x: np.ndarray, gate_base: np.ndarray, gate_offset: int, s_gate_b: int,
                      y: np.ndarray, B: int, N: int, D: int, dtype: str = "bf16",
                      rows: Optional[Sequence[int]] = None, threads: int = 1):
    """``x + gate*y`` with per-op storage rounding; returns (row_ids, out)."""
    lib = _lib_handle()
    xf, yf, gf = _u16(x).reshape(-1), _u16(y).reshape(-1), _u16(gate_base).reshape(-1)
    idx, runs = _segments(rows, B * N)
    out = np.zeros((idx.size, D), dtype=np.uint16)
    pos = {int(r): i for i, r in enumerate(idx)}

    def one(piece):
        b0, e0 = piece
        lib.oracle_residual_gate_add(out[pos[b0]:].ctypes.data, xf.ctypes.data,
                                     gf.ctypes.data + 2 * gate_offset, s_gate_b, yf.ctypes.data,
                                     B, N, D, DTYPE_CODE[dtype], b0, e0)

    _run(_split_runs(runs, threads), one, threads)
    return idx, out


def residual_gate_ln_modulate(x: np.ndarray, gate_base: np.ndarray, gate_offset: int, s_gate_b: int,
                              y: np.ndarray, B: int, N: int, D: int, scale_base: np.ndarray,
                              scale_offset: int, s_scale_b: int, shift_base: np.ndarray,
                              shift_offset: int, s_shift_b: int, eps: float, dtype: str = "bf16",
                              rows: Optional[Sequence[int]] = None, threads: int = 1):
    """``r = x + gate*y``, then ``LN(r)*(1+scale)+shift`` of r as stored: the
    Fused Kernels page's scale_residual_norm_scale_shift (Kernel inventory,
    Normalization table) is exactly the gate-add chain followed by the
    LN+modulate chain, so this is their composition.  Returns (row_ids, r, out)."""
    ids, r = residual_gate_add(x, gate_base, gate_offset, s_gate_b, y, B, N, D, dtype, rows=rows,
                               threads=threads)
    out = np.empty_like(r)
    # LN+modulate row by row of r (rows of one sample share the scale / shift row)
    for b in np.unique(ids // N):
        sel = np.nonzero(ids // N == b)[0]
        rb = np.ascontiguousarray(r[sel])
        _, ob = ln_modulate(rb, 1, sel.size, D, (sel.size * D, D, 1), scale_base,
                            scale_offset + int(b) * s_scale_b, 0, shift_base,
                            shift_offset + int(b) * s_shift_b, 0, eps, dtype, threads=threads)
        out[sel] = ob
    return ids, r, out


NORM_CODE = {"layer": 0, "rms": 1}


def norm_scale_shift(norm: str, x_base: np.ndarray, B: int, N: int, D: int,
                     strides: Tuple[int, int, int], scale_base: np.ndarray, scale_offset: int,
                     s_scale_b: int, s_scale_n: int, shift_base: np.ndarray, shift_offset: int,
                     s_shift_b: int, s_shift_n: int, eps: float, dtype: str = "bf16",
                     gate: Optional[Tuple[np.ndarray, int, int, int, int]] = None,
                     y: Optional[np.ndarray] = None, rows: Optional[Sequence[int]] = None,
                     threads: int = 1, return_stats: bool = False):
    """LayerNorm (``norm="layer"``) or RMSNorm (``"rms"``), no affine, then
    ``* (1 + scale) + shift``, optionally after the residual gate-add
    ``r = x + gate * y`` (Fused Kernels page, Normalization table:
    rmsnorm_scale_shift, scale_residual_norm_scale_shift; request-gated
    fusion table: per-token [B, S, 1] gates, strided [B, S, 6D] chunk views).

    Element (b, n, d) of x sits at ``b*sxB + n*sxN + d*sxD`` of ``x_base``;
    of scale at ``scale_offset + b*s_scale_b + n*s_scale_n + d`` (shift
    likewise).  ``gate = (base, offset, s_b, s_n, s_d)`` places gate
    (b, n, d) at ``offset + b*s_b + n*s_n + d*s_d`` (s_d = 0 for a per-token
    scalar); y is contiguous (B, N, D).  Returns ``(row_ids, out)``, or
    ``(row_ids, r, out)`` with a gate; with ``return_stats`` also the per-row
    binary32 mean (0 for RMSNorm) and rstd."""
    lib = _lib_handle()
    xb, sb, hb = _u16(x_base).reshape(-1), _u16(scale_base).reshape(-1), _u16(shift_base).reshape(-1)
    idx, runs = _segments(rows, B * N)
    out = np.zeros((idx.size, D), dtype=np.uint16)
    r_out = np.zeros((idx.size, D), dtype=np.uint16) if gate is not None else None
    mean = np.zeros(idx.size, dtype=np.float32)
    rstd = np.zeros(idx.size, dtype=np.float32)
    pos = {int(r): i for i, r in enumerate(idx)}
    sxB, sxN, sxD = strides
    if gate is not None:
        gb, goff, sgb, sgn, sgd = gate
        gb = _u16(gb).reshape(-1)
        yb = _u16(y).reshape(-1)
        if yb.size < B * N * D:
            raise ValueError("y must hold B*N*D values")

    def one(piece):
        b0, e0 = piece
        i0 = pos[b0]
        if gate is not None:
            gargs = (gb.ctypes.data + 2 * goff, sgb, sgn, sgd, yb.ctypes.data)
            rptr = r_out[i0:].ctypes.data
        else:
            gargs, rptr = (None, 0, 0, 0, None), None
        rc = lib.oracle_norm_scale_shift(rptr, out[i0:].ctypes.data, NORM_CODE[norm], xb.ctypes.data,
                                         B, N, D, sxB, sxN, sxD, *gargs,
                                         sb.ctypes.data + 2 * scale_offset, s_scale_b, s_scale_n,
                                         hb.ctypes.data + 2 * shift_offset, s_shift_b, s_shift_n, eps,
                                         DTYPE_CODE[dtype], b0, e0, mean[i0:].ctypes.data,
                                         rstd[i0:].ctypes.data)
        if rc:
            raise ValueError(f"oracle_norm_scale_shift rejected its arguments ({rc})")

    _run(_split_runs(runs, threads), one, threads)
    res = (idx, out) if gate is None else (idx, r_out, out)
    return res + (mean, rstd) if return_stats else res


def qk_rmsnorm(x: np.ndarray, Dh: int, w: np.ndarray, eps: float, dtype: str = "bf16",
               rows: Optional[Sequence[int]] = None, threads: int = 1):
    """Per-head RMSNorm with a weight on a (rows, Dh) tensor (Fused Kernels
    page, Normalization table: qk_rmsnorm_native); returns (row_ids, out)."""
    lib = _lib_handle()
    xf = _u16(x).reshape(-1)
    nrows = xf.size // Dh
    w = _u16(w).reshape(-1)
    idx, runs = _segments(rows, nrows)
    out = np.zeros((idx.size, Dh), dtype=np.uint16)
    pos = {int(r): i for i, r in enumerate(idx)}

    def one(piece):
        b0, e0 = piece
        rc = lib.oracle_qk_rmsnorm(out[pos[b0]:].ctypes.data, xf.ctypes.data, nrows, Dh, w.ctypes.data,
                                   eps, DTYPE_CODE[dtype], b0, e0)
        if rc:
            raise ValueError(f"oracle_qk_rmsnorm rejected its arguments ({rc})")

    _run(_split_runs(runs, threads), one, threads)
    return idx, out


def temb_table_slices(table: np.ndarray, table_dtype: str, temb: np.ndarray, temb_dtype: str,
                      B: int, S: int, K: int, D: int) -> np.ndarray:
    """``(table + temb.float()).chunk(K)`` as K contiguous binary32 slices
    (Fused Kernels page, adaLN modulation and gating table: temb_table_slices).
    table (K, D) and temb (B, S, K, D) hold uint16 patterns (bf16 / fp16) or
    float32.  Returns a float32 array (K, B, S, D)."""
    def arr(a, dt):
        return np.ascontiguousarray(a, dtype=np.float32 if dt == "fp32" else np.uint16).reshape(-1)
    t, e = arr(table, table_dtype), arr(temb, temb_dtype)
    if t.size != K * D or e.size != B * S * K * D:
        raise ValueError("table must hold K*D values and temb B*S*K*D")
    out = np.zeros((K, B, S, D), dtype=np.float32)
    rc = _lib_handle().oracle_temb_table_slices(out.ctypes.data, B * S * D, t.ctypes.data,
                                                ANY_DTYPE_CODE[table_dtype], e.ctypes.data,
                                                ANY_DTYPE_CODE[temb_dtype], B, S, K, D)
    if rc:
        raise ValueError("oracle_temb_table_slices rejected its arguments")
    return out


def quant_e4m3(y: np.ndarray, qscale: float, dtype: str = "bf16") -> np.ndarray:
    """Static FP8 quantisation of storage values: e4m3(value(y) / qscale),
    binary32 division, round to nearest even, saturating at 448 (the
    Quantized layout producers table's static FP8 output).  Returns uint8."""
    yf = np.ascontiguousarray(_u16(y))
    out = np.zeros(yf.shape, dtype=np.uint8)
    _lib_handle().oracle_quant_e4m3(out.ctypes.data, yf.ctypes.data, yf.size, float(np.float32(qscale)),
                                    DTYPE_CODE[dtype])
    return out


def e4m3(f: np.ndarray) -> np.ndarray:
    """binary32 values -> e4m3 codes (round to nearest even, saturating)."""
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint8)
    _lib_handle().oracle_f32_to_e4m3_array(f.ctypes.data, out.ctypes.data, f.size)
    return out


def ln_modulate_fp8(x_base: np.ndarray, B: int, N: int, D: int, strides: Tuple[int, int, int],
                    scale_base: np.ndarray, scale_offset: int, s_scale_b: int,
                    shift_base: np.ndarray, shift_offset: int, s_shift_b: int, eps: float, qscale: float,
                    dtype: str = "bf16", rows: Optional[Sequence[int]] = None, threads: int = 1):
    """LayerNorm + adaLN modulate written as static FP8: ln_modulate's
    storage output quantised by quant_e4m3 (Fused Kernels page, Quantized
    layout producers table: flux2_layernorm_modulate_fp8_quant).  Returns
    (row_ids, uint8 codes (rows, D))."""
    ids, y = ln_modulate(x_base, B, N, D, strides, scale_base, scale_offset, s_scale_b, shift_base, shift_offset,
                         s_shift_b, eps, dtype, rows=rows, threads=threads)
    return ids, quant_e4m3(y, qscale, dtype)


def bias_gelu_tanh(x: np.ndarray, bias: np.ndarray, rows_total: int, width: int,
                   dtype: str = "bf16", rows: Optional[Sequence[int]] = None,
                   threads: int = 1):
    """``gelu_tanh(round(x + bias))`` rounded to storage; returns (row_ids, out)."""
    lib = _lib_handle()
    xf, bf = _u16(x).reshape(-1), _u16(bias).reshape(-1)
    idx, runs = _segments(rows, rows_total)
    out = np.zeros((idx.size, width), dtype=np.uint16)
    pos = {int(r): i for i, r in enumerate(idx)}
    gelu_table(dtype)  # build the table once, before any threads start

    def one(piece):
        b0, e0 = piece
        lib.oracle_bias_gelu_tanh(out[pos[b0]:].ctypes.data, xf.ctypes.data, bf.ctypes.data,
                                  rows_total, width, DTYPE_CODE[dtype], b0, e0)

    _run(_split_runs(runs, threads), one, threads)
    return idx, out


_tables = {}


def gelu_table(dtype: str = "bf16") -> np.ndarray:
    """All 65536 outputs ``round16(G(v))`` indexed by the pattern of v."""
    if dtype not in _tables:
        t = np.zeros(65536, dtype=np.uint16)
        _lib_handle().oracle_gelu_table(t.ctypes.data, DTYPE_CODE[dtype])
        # also warm the C side's own copy used by oracle_bias_gelu_tanh
        one = np.zeros(1, dtype=np.uint16)
        _lib_handle().oracle_bias_gelu_tanh(one.ctypes.data, one.ctypes.data, one.ctypes.data,
                                            1, 1, DTYPE_CODE[dtype], 0, 1)
        _tables[dtype] = t
    return _tables[dtype]


# --------------------------------------------------------------------------
# helpers used by the oracle's own pins
# --------------------------------------------------------------------------

def to16(f: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    _lib_handle().oracle_f32_to_16(f.ctypes.data, out.ctypes.data, f.size, DTYPE_CODE[dtype])
    return out


def from16(h: np.ndarray, dtype: str = "bf16") -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _lib_handle().oracle_16_to_f32(h.ctypes.data, out.ctypes.data, h.size, DTYPE_CODE[dtype])
    return out


def rsqrt_cr(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(x)
    _lib_handle().oracle_rsqrt_cr_array(x.ctypes.data, out.ctypes.data, x.size)
    return out


def row_sumsq(row: np.ndarray, lanes: int = 128) -> float:
    """RMSNorm sum of squares of one binary32 row on the canonical lane DAG."""
    row = np.ascontiguousarray(row, dtype=np.float32)
    ss = np.zeros(1, dtype=np.float32)
    if _lib_handle().oracle_row_sumsq(row.ctypes.data, row.size, lanes, ss.ctypes.data):
        raise ValueError("bad row length / lane count")
    return float(ss[0])


def row_stats(row: np.ndarray, lanes: int = 128) -> Tuple[float, float]:
    """(mean, m2) of one binary32 row on the canonical lane DAG."""
    row = np.ascontiguousarray(row, dtype=np.float32)
    m = np.zeros(1, dtype=np.float32)
    q = np.zeros(1, dtype=np.float32)
    rc = _lib_handle().oracle_row_stats(row.ctypes.data, row.size, lanes, m.ctypes.data,
                                        q.ctypes.data)
    if rc:
        raise ValueError("bad row length / lane count")
    return float(m[0]), float(q[0])
