"""Writes oracle_regression.json: small cases of every oracle chain (inputs
from the seeded generator, outputs from the oracle), as 16-bit patterns in
hex.  The pages print no worked example with values, so these fixtures are
regression fixtures of the pinned oracle (they catch an unintended change to
its arithmetic), not independent pins.  Run from the repository root:

    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def hx(a):
    a = np.asarray(a)
    if a.dtype == np.float32:
        a = a.view(np.uint32)
    return [format(int(v), "x") for v in a.reshape(-1)]


def cases():
    out = {}
    B, N, D = 2, 3, 12
    x = synth.normal_bits(101, B * N * D, 0.3, 1).reshape(B, N, D)
    t = synth.normal_bits(102, B * 2 * D, 0, 0.2)
    y = synth.normal_bits(103, B * N * D, 0, 1).reshape(B, N, D)
    gs = synth.normal_bits(104, B * N, 0, 0.5)
    for norm in ("layer", "rms"):
        _, o = oracle.norm_scale_shift(norm, x, B, N, D, (N * D, D, 1), t, D, 2 * D, 0, t, 0, 2 * D, 0, 1e-6)
        _, r, og = oracle.norm_scale_shift(norm, x, B, N, D, (N * D, D, 1), t, D, 2 * D, 0, t, 0, 2 * D, 0, 1e-6,
                                           gate=(gs, 0, N, 1, 0), y=y)
        out[f"{norm}_modulate"] = {"x": hx(x), "table": hx(t), "out": hx(o)}
        out[f"{norm}_gated_per_token"] = {"x": hx(x), "y": hx(y), "gate": hx(gs), "table": hx(t), "r": hx(r),
                                          "out": hx(og)}
    q = synth.normal_bits(105, 4 * 8, 0, 2).reshape(4, 8)
    w = synth.normal_bits(106, 8, 1, 0.05)
    bq = synth.normal_bits(107, 8, 0, 0.05)
    out["qk_layernorm"] = {"q": hx(q), "w": hx(w), "b": hx(bq), "out": hx(oracle.qk_head_layernorm(q, 8, w, bq, 1e-6)[1])}
    out["qk_rmsnorm"] = {"q": hx(q), "w": hx(w), "out": hx(oracle.qk_rmsnorm(q, 8, w, 1e-6)[1])}
    g = synth.normal_bits(108, B * D, 0, 0.1).reshape(B, 1, D)
    out["residual_gate_add"] = {"x": hx(x), "gate": hx(g), "y": hx(y),
                                "out": hx(oracle.residual_gate_add(x, g, 0, D, y, B, N, D)[1])}
    for dt in ("bf16", "fp16"):
        xd = synth.normal_bits(109, 2 * 16, 0, 2, dt).reshape(2, 16)
        bd = synth.normal_bits(110, 16, 0, 0.1, dt)
        out[f"bias_gelu_{dt}"] = {"x": hx(xd), "bias": hx(bd), "out": hx(oracle.bias_gelu_tanh(xd, bd, 2, 16, dt)[1])}
    tab = (synth.normal_bits(111, 3 * 8, 0, 0.05).astype(np.uint32) << 16).view(np.float32).reshape(3, 8)
    temb = synth.normal_bits(112, 2 * 3 * 8, 0, 1).reshape(1, 2, 3, 8)
    out["temb_table_slices"] = {"table_f32": hx(tab), "temb": hx(temb),
                                "out_f32": hx(oracle.temb_table_slices(tab, "fp32", temb, "bf16", 1, 2, 3, 8))}
    _, q8 = oracle.ln_modulate_fp8(x, B, N, D, (N * D, D, 1), t, D, 2 * D, t, 0, 2 * D, 1e-6, 0.01)
    out["ln_modulate_fp8"] = {"x": hx(x), "table": hx(t), "qscale": 0.01, "out_e4m3": hx(q8)}
    return out


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(cases(), f, indent=0, sort_keys=True)
    print("wrote", path)
