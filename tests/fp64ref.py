"""Double-precision references used to pin the oracle (test helpers).

Nothing here reuses the oracle's code: storage rounding is done by scaling
with powers of two and ``np.rint`` (IEEE round-half-even to an integer), not
by bit manipulation, and the statistics are a two-pass mean / variance in
float64.
"""
import numpy as np

# (significand bits p, minimum normal exponent, maximum finite value)
FORMATS = {"bf16": (8, -126, float.fromhex("0x1.fep127")),
           "fp16": (11, -14, 65504.0)}


def round_to16(v, dtype="bf16"):
    """Round real values (given exactly as float64) to the nearest bf16/fp16
    value, ties to even; overflow -> inf.  Returns float64."""
    p, emin, vmax = FORMATS[dtype]
    v = np.asarray(v, dtype=np.float64)
    out = np.array(v, dtype=np.float64, copy=True)
    fin = np.isfinite(v) & (v != 0)
    a = np.abs(v[fin])
    _, ex = np.frexp(a)                      # a = m * 2**ex, m in [0.5, 1)
    e = np.maximum(ex - 1, emin)             # exponent of the leading bit
    scale = np.ldexp(1.0, (p - 1) - e)
    r = np.rint(a * scale) / scale           # exact scalings by powers of two
    r = np.where(r > vmax, np.inf, r)
    out[fin] = np.copysign(r, v[fin])
    return out


def bits16(v, dtype="bf16"):
    """Bit patterns of float64 values that are exactly representable."""
    v = np.asarray(v, dtype=np.float64)
    if dtype == "fp16":
        return v.astype(np.float16).view(np.uint16)
    return (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def value16(h, dtype="bf16"):
    h = np.asarray(h, dtype=np.uint16)
    if dtype == "fp16":
        return h.view(np.float16).astype(np.float64)
    with np.errstate(invalid="ignore"):
        return (h.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def ordered(h, dtype="bf16"):
    """Map patterns to integers whose difference counts ulps (+0 == -0)."""
    h = np.asarray(h, dtype=np.uint16).astype(np.int64)
    mag = h & 0x7FFF
    return np.where(h & 0x8000, -mag, mag)


def ulp_diff(a, b, dtype="bf16"):
    return np.abs(ordered(a, dtype) - ordered(b, dtype))


def ln_fp64(xv, eps):
    """Two-pass LayerNorm in float64 over the last axis (eps given as float32)."""
    x = np.asarray(xv, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + float(np.float32(eps)))
    return (x - mean) * rstd, mean, rstd


def ln_modulate_fp64(xv, sc, sh, eps, dtype="bf16"):
    """fp64 statistics, the chain's storage rounding points: y, 1+scale,
    y*op and p+shift each rounded once to the storage type."""
    y, _, _ = ln_fp64(xv, eps)
    y = round_to16(y, dtype)
    op = round_to16(1.0 + np.asarray(sc, np.float64), dtype)
    p = round_to16(y * op, dtype)
    return round_to16(p + np.asarray(sh, np.float64), dtype)
