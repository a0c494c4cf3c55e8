"""The oracle's pins catch plausible mistakes.

Each case below plants one mistake in a temporary copy of ``oracle/oracle.c``
(a dropped term, a wrong sign or index, a transposed operand, a missing
rounding, a wrong constant), builds it, and runs the pin suite against it:
at least one pin must fail.  The real oracle is untouched.

Three mistakes change only the *order* of roundings inside the canonical
lane DAG (the fold order, the operand order of the symmetric combine, the
element-to-lane assignment).  They leave every value within the fp32 error
bound, so value pins cannot see them; they are caught by the exact-row pins
where they turn exact steps into inexact ones, and otherwise only by the
bit-exact comparison with the independently written CUDA path.  They are
listed in ``ORDER_ONLY`` and checked to stay within the value pins.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_ln as ln
import test_oracle_qk_gate_gelu as qg
import test_oracle_rms as rm
import test_oracle_fp8 as f8
import test_oracle_temb as tb
import test_oracle_rsqrt as rs
import test_oracle_conversions as cv

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "drop_delta_sq_term": ("o.m2 = fmaf(dda, coef, m2s);", "o.m2 = m2s;"),
    "delta_sign": ("float delta = b.mean - a.mean;", "float delta = a.mean - b.mean;"),
    "welford_old_mean": ("float t = v - mean;", "float t = v - s->mean;"),
    "welford_count_off_by_one": ("float r = 1.0f / c1;", "float r = 1.0f / (c1 + 1.0f);"),
    "unguarded_coef": ("float coef = (n == 0.0f) ? 0.0f : b.cnt / n;", "float coef = b.cnt / n;"),
    "sample_variance": ("float var = m2 / (float)D;", "float var = m2 / (float)(D - 1);"),
    "eps_dropped": ("return oracle_rsqrt_cr(var + eps);", "return oracle_rsqrt_cr(var);"),
    "rsqrt_uncorrected": ("    for (int it = 0; it < 4; ++it) {\n        float up",
                          "    r = (float)(1.0f / sqrtf(x)); return r;\n    for (int it = 0; it < 4; ++it) {\n        float up"),
    "y_not_rounded": ("float y = round16(rstd * centered, dtype);", "float y = rstd * centered;"),
    "one_plus_scale_not_rounded": ("float op = round16(1.0f + load16(sc[d], dtype), dtype);",
                                   "float op = 1.0f + load16(sc[d], dtype);"),
    "product_not_rounded": ("float p = round16(y * op, dtype);", "float p = y * op;"),
    "shift_scale_swapped": ("const uint16_t *sc = scale + b * s_scale_b + n * s_scale_n, *sh = shift + b * s_shift_b + n * s_shift_n;",
                            "const uint16_t *sh = scale + b * s_scale_b + n * s_scale_n, *sc = shift + b * s_shift_b + n * s_shift_n;"),
    "tail_lanes_push_zeros": ("for (int64_t j = l; j < nvec; j += L)\n            for (int e = 0; e < 4; ++e) welford_push(&st[l], x[4 * j + e]);",
                              "for (int64_t j = l; j < ((nvec + L - 1) / L) * L; j += L)\n            for (int e = 0; e < 4; ++e) welford_push(&st[l], j < nvec ? x[4 * j + e] : 0.0f);"),
    "qk_w_b_swapped": ("store16(fmaf(load16(w[d], dtype), u, load16(bias[d], dtype)), dtype);",
                       "store16(fmaf(load16(bias[d], dtype), u, load16(w[d], dtype)), dtype);"),
    "gate_product_not_rounded": ("float gy = round16(load16(g, dtype) * load16(yv, dtype), dtype);",
                                 "float gy = load16(g, dtype) * load16(yv, dtype);"),
    "rms_subtracts_mean": ("            mean = 0.0f;\n            rstd = rms_rstd(",
                           "            { float m2_; row_stats(v, D, 128, &mean, &m2_); }\n            rstd = rms_rstd("),
    "rms_divisor_d_minus_1": ("float ms = ss / (float)D;", "float ms = ss / (float)(D - 1);"),
    "rms_eps_dropped": ("return oracle_rsqrt_cr(ms + eps);", "return oracle_rsqrt_cr(ms);"),
    "rms_abs_not_square": ("float sq = x[4 * j + e] * x[4 * j + e];", "float sq = fabsf(x[4 * j + e]);"),
    "rms_fold_drops_upper": ("nx[l] = st[l & ~o] + st[l | o];", "nx[l] = st[l & ~o];"),
    "per_token_scale_row_index": ("scale + b * s_scale_b + n * s_scale_n,", "scale + b * s_scale_b + b * s_scale_n,"),
    "per_token_gate_row_ignored": ("const uint16_t *g = gate + b * s_gate_b + n * s_gate_n;",
                                   "const uint16_t *g = gate + b * s_gate_b;"),
    "gate_elem_stride_ignored": ("gate_add(v[d], g[d * s_gate_d], y[r * D + d], dtype)",
                                 "gate_add(v[d], g[d], y[r * D + d], dtype)"),
    "gated_norm_reads_x": ("for (int64_t d = 0; d < D; ++d) v[d] = gate_add(",
                           "for (int64_t d = 0; d < D && 0; ++d) v[d] = gate_add("),
    "qk_rms_weight_dropped": ("store16(load16(w[d], dtype) * u, dtype);", "store16(u, dtype);"),
    "temb_chunk_major_layout": ("load_any(temb, (bs * K + k) * D + d, temb_dtype)",
                                "load_any(temb, (k * B * S + bs) * D + d, temb_dtype)"),
    "temb_table_row_zero": ("load_any(table, k * D + d, table_dtype)", "load_any(table, d, table_dtype)"),
    "e4m3_ties_away_from_zero": ("if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;",
                                 "if (frac >= 0.5) r += 1.0;"),
    "e4m3_no_saturation": ("if (a >= 448.0) return sign | 0x7e;", "if (a >= 4480.0) return sign | 0x7e;"),
    "e4m3_subnormal_quantum": ("if (ex < -6) ex = -6;", "if (ex < -7) ex = -7;"),
    "quant_by_reciprocal": ("f32_to_e4m3_sat(load16(y[i], dtype) / qscale)",
                            "f32_to_e4m3_sat(load16(y[i], dtype) * (1.0f / qscale))"),
    "temb_slice_stride_ignored": ("out[k * s_out_k + bs * D + d] =", "out[k * B * S * D / K + bs * D + d] ="),
    "gelu_constant_typo": ("const long double k1 = 0.044715L;", "const long double k1 = 0.04715L;"),
    "gelu_sign": ("long double g = v / (1.0L + expl(-2.0L * z));", "long double g = v / (1.0L + expl(2.0L * z));"),
    "gelu_bias_dropped": ("uint16_t v = store16(load16(x[r * width + c], dtype) + load16(bias[c], dtype), dtype);",
                          "uint16_t v = x[r * width + c];"),
    "bf16_round_half_up": ("return (uint16_t)((u + 0x7fffu + lsb) >> 16);", "return (uint16_t)((u + 0x8000u) >> 16);"),
    "fp16_subnormal_truncated": ("if (rem > half || (rem == half && (q & 1u))) ++q;", "(void)rem; (void)half;"),
}

ORDER_ONLY = {
    "fold_order_reversed": ("static const int order128[7] = {16, 8, 4, 2, 1, 64, 32};",
                            "static const int order128[7] = {1, 2, 4, 8, 16, 32, 64};"),
    "combine_operands_transposed": ("nx[l] = chan_combine(st[l & ~o], st[l | o]);",
                                    "nx[l] = chan_combine(st[l | o], st[l & ~o]);"),
    "blocked_lane_assignment": ("for (int64_t j = l; j < nvec; j += L)\n            for (int e = 0; e < 4; ++e) welford_push",
                                "for (int64_t j = l * ((nvec + L - 1) / L); j < nvec && j < (l + 1) * ((nvec + L - 1) / L); ++j)\n            for (int e = 0; e < 4; ++e) welford_push"),
    "rms_square_fused_into_sum": ("float sq = x[4 * j + e] * x[4 * j + e];\n                st[l] = st[l] + sq;",
                                  "st[l] = fmaf(x[4 * j + e], x[4 * j + e], st[l]);"),
    "qk_rms_on_128_lanes": ("rms_rstd(row_sumsq(v, Dh, 32), Dh, eps)", "rms_rstd(row_sumsq(v, Dh, 128), Dh, eps)"),
}


def _pins():
    """(name, callable) for a fast subset of every pin family."""
    P = []
    for D in (12, 516, 2240, 4096):
        P.append((f"ln_fp64_{D}", lambda D=D: ln.test_ln_within_one_ulp_of_fp64_two_pass(None, D, "bf16")))
    P.append(("ln_fp64_fp16", lambda: ln.test_ln_within_one_ulp_of_fp64_two_pass(None, 2240, "fp16")))
    P.append(("ln_offset", lambda: ln.test_ln_offset_rows_within_fp32_mean_error(None, 516, "bf16")))
    P.append(("chain", lambda: ln.test_full_chain_vs_fp64_statistics(None, 2240)))
    for D in (512, 4096):
        P.append((f"exact_{D}", lambda D=D: ln.test_exact_rows_equal_rationals(None, D)))
    P.append(("exact_tail", lambda: ln.test_exact_rows_tail_chunk_2240(None)))
    P.append(("constant", lambda: ln.test_constant_rows(None, 2240)))
    P.append(("scale_m1", lambda: ln.test_scale_minus_one_returns_shift(None, 2240)))
    P.append(("tail_def", lambda: ln.test_modulate_tail_matches_definition(None, "bf16")))
    P.append(("negation", lambda: ln.test_negation_symmetry(None, 2240)))
    P.append(("pow2", lambda: ln.test_power_of_two_scaling_invariance(None, 2240)))
    P.append(("qk_plain", lambda: qg.test_qk_plain_ln_within_one_ulp(None, 128, "bf16")))
    P.append(("qk_plain_short", lambda: qg.test_qk_plain_ln_within_one_ulp(None, 100, "bf16")))
    P.append(("qk_affine", lambda: qg.test_qk_affine_within_rounding_bound(None, "bf16")))
    P.append(("gate", lambda: qg.test_gate_add_equals_single_rounding_definition(None, "bf16")))
    P.append(("gate_fp16", lambda: qg.test_gate_add_equals_single_rounding_definition(None, "fp16")))
    P.append(("gelu_special", lambda: qg.test_gelu_special_points(None, "bf16")))
    P.append(("gelu_sum", lambda: qg.test_bias_gelu_rounds_the_sum_once(None, "bf16")))
    P.append(("gelu_table", lambda: qg.test_gelu_table_matches_high_precision(None, "bf16")))
    P.append(("rsqrt", lambda: rs.test_rsqrt_matches_100bit_reference(None)))
    for D in (12, 2240, 5120):
        P.append((f"rms_fp64_{D}", lambda D=D: rm.test_rms_within_one_ulp_of_fp64(None, D, "bf16")))
    P.append(("rms_exact", lambda: rm.test_exact_rows_give_half(None, 2240, "bf16", (3, 3, 3, 1, 1, 1, 1, 1), 0.0)))
    P.append(("rms_exact_eps", lambda: rm.test_exact_rows_give_half(None, 512, "bf16", (3, 3, 3, 1, 1, 1, 0, 0), 0.25)))
    P.append(("rms_signs", lambda: rm.test_sign_flips_flip_only_those_outputs(None, 516)))
    P.append(("rms_tail_def", lambda: rm.test_modulate_tail_matches_definition(None, "bf16")))
    for norm in ("layer", "rms"):
        P.append((f"gated_{norm}", lambda norm=norm: rm.test_gated_mode_is_gate_add_then_norm(None, norm)))
        P.append((f"per_token_{norm}", lambda norm=norm: rm.test_per_token_rows_and_gates_equal_one_row_calls(None, norm)))
    P.append(("qk_rms", lambda: rm.test_qk_rms_within_rounding_bound(None, 128, "bf16")))
    P.append(("qk_rms_exact", lambda: rm.test_qk_rms_exact_rows(None, 64)))
    P.append(("temb_add", lambda: tb.test_slices_equal_numpy_binary32_add(None, "fp32", "bf16")))
    P.append(("temb_order", lambda: tb.test_slice_order_and_broadcast(None)))
    P.append(("e4m3_round_trip", lambda: f8.test_every_code_round_trips(None)))
    P.append(("e4m3_ties", lambda: f8.test_ties_saturation_nan_and_zero(None)))
    P.append(("e4m3_torch", lambda: f8.test_quantiser_matches_torch_on_every_pattern(None, "bf16", 0.37)))
    P.append(("e4m3_div_ties", lambda: f8.test_exact_ties_after_division(None)))
    P.append(("bf16_encode", lambda: cv.test_bf16_encode_vs_torch(None)))
    P.append(("fp16_encode", lambda: cv.test_fp16_encode_vs_numpy(None)))
    return P


def _build_mutant(tmp_path, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique/found"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", *oracle.CFLAGS, str(path), "-o", str(so), "-lm"], check=True,
                   capture_output=True)
    return str(so)


def _failures(so, stop_first=False):
    failed = []
    with oracle.loaded_from(so):
        for pname, fn in _pins():
            try:
                fn()
            except (AssertionError, ValueError, IndexError):
                failed.append(pname)
                if stop_first:
                    break
    return failed


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(oracle_lib, tmp_path, name):
    pytest.importorskip("mpmath")
    so = _build_mutant(tmp_path, name, *MUTANTS[name])
    assert _failures(so, stop_first=True), f"no pin caught mutant {name}"


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(ORDER_ONLY))
def test_order_only_mutants_keep_values(oracle_lib, tmp_path, name):
    """Order-only mistakes stay inside every value pin except, possibly, the
    exact-row ones; the independently written CUDA path is their check."""
    pytest.importorskip("mpmath")
    so = _build_mutant(tmp_path, name, *ORDER_ONLY[name])
    failed = set(_failures(so))
    print(name, "caught by", sorted(failed))
    assert failed <= {"exact_512", "exact_4096", "exact_tail"}, failed
