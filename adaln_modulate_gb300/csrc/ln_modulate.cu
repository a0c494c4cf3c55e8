// Fused LayerNorm (no affine) + adaLN modulate for sm_103a.
//
// Follows the "layernorm_modulate" entry of the SGLang Diffusion "Fused
// Kernels" page (Normalization table; "Numerical contracts and quality
// tiers": serial Welford per thread, guarded reciprocal, fixed fold tree)
// and PR #34015 "实现拆解" 1 (vec4 chunks, (D+511)/512 iterations, tail lanes
// whose vec index reaches D/4 skip and enter the fold with a smaller count;
// pass 2: y rounded to the storage type, 1 + scale rounded, product rounded,
// fp32 add of shift rounded by the store).
//
// The rounding DAG is fixed by 128 LOGICAL lanes; the kernels below map
// them onto threads differently but compute the same bits:
//   ln_rows_kernel    contiguous rows, one warp per row, 4 logical lanes per
//                     thread (lanes l0 + 8s, one 8-byte access each per
//                     512-element step), row held in registers;
//   ln_tokens_kernel  the (B, N, D) view of a contiguous (B, D, N) tensor
//                     (tokens contiguous): a CTA takes 8 consecutive tokens,
//                     one thread per logical lane for all 8, 16-byte
//                     cp.async of each d-row (8 tokens) into thread-private
//                     shared memory, writes the output contiguous;
//   ln_generic_kernel any strides, one CTA of 128 threads per row, scalar
//                     loads; the arithmetic is plain binary32 code.
//
// The same kernels serve the RMSNorm chain (rmsnorm_scale_shift of the
// Normalization table: the lanes sum squares instead of running Welford,
// the output pass is the LayerNorm's with mean 0), per-token modulation
// rows (the strided [B, S, 6D] chunk views of the request-gated fusion
// table) and the residual gate-add in front (scale_residual_norm_scale_shift,
// with a per-sample gate row or a per-token [B, S, 1] gate), and the static
// FP8 output of the Quantized layout producers table
// (flux2_layernorm_modulate_fp8_quant: e4m3(y / scale) of every output y);
// the tokens kernels take only the LayerNorm with per-sample rows, no gate
// and storage output.
#include "ln_common.cuh"

namespace adaln {

// The contiguous-rows kernel moves every logical lane's vec4 chunk with one
// 8-byte access, so every row start of x, out, scale and shift (and with a
// gate of y, r_out and the gate rows) must be 8-byte aligned.  Strides of
// size-1 dimensions are never used and are ignored.
bool ln_rows_ok(const LnArgs &a) {
    const bool base = ln_aligned(a.x, 8) && ln_aligned(a.out, 8) && ln_aligned(a.scale, 8) &&
                      ln_aligned(a.shift, 8) && (a.N == 1 || ln_mult(a.sxN, 4)) &&
                      (a.B == 1 || (ln_mult(a.sxB, 4) && ln_mult(a.s_scale_b, 4) && ln_mult(a.s_shift_b, 4))) &&
                      (a.N == 1 || (ln_mult(a.s_scale_n, 4) && ln_mult(a.s_shift_n, 4)));
    if (!base || !a.gate) return base;
    if (!ln_aligned(a.y, 8) || !ln_aligned(a.r_out, 8)) return false;
    // a per-token scalar gate is read one value at a time
    return a.s_gate_d == 0 || (ln_aligned(a.gate, 8) && (a.B == 1 || ln_mult(a.s_gate_b, 4)) &&
                               (a.N == 1 || ln_mult(a.s_gate_n, 4)));
}

int ln_modulate_path(const LnArgs &a) {
    const int64_t ni = (a.D + 511) / 512;
    // the static FP8 output has rows kernels for the gate-free LayerNorm only
    const bool rows_kind = !a.qscale || (a.norm == 0 && !a.gate);
    if (rows_kind && a.sxD == 1 && ni <= kRowsMaxNI && ln_rows_ok(a)) return LN_PATH_ROWS;
    // tokens contiguous (LayerNorm, one scale / shift row per sample, no
    // gate, storage output): each d-row of 8 tokens is one 16-byte copy
    const bool per_sample = a.s_scale_n == 0 && a.s_shift_n == 0;
    if (a.norm == 0 && !a.gate && !a.qscale && per_sample && a.sxN == 1 && a.sxD != 1 && a.N > 1 && ni <= kTokensMaxNI &&
        ln_aligned(a.x, 16) && ln_mult(a.sxD, 8) &&
        (a.B == 1 || (ln_mult(a.sxB, 8) && ln_mult(a.s_scale_b, 4) && ln_mult(a.s_shift_b, 4))) &&
        ln_aligned(a.out, 8) && ln_aligned(a.scale, 8) && ln_aligned(a.shift, 8))
        return LN_PATH_TOKENS;
    return LN_PATH_GENERIC;
}

cudaError_t launch_norm_scale_shift(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    switch (ln_modulate_path(a)) {
        case LN_PATH_ROWS: {
            using RowsFn = cudaError_t (*)(const LnArgs &, bool, cudaStream_t, const DeviceInfo &);
            static const RowsFn fns[2][2][2] = {  // [norm][gate][dtype]
                {{rows_ln_bf16, rows_ln_fp16}, {rows_ln_gate_bf16, rows_ln_gate_fp16}},
                {{rows_rms_bf16, rows_rms_fp16}, {rows_rms_gate_bf16, rows_rms_gate_fp16}}};
            if (a.qscale) return dtype == 0 ? rows_ln_fp8_bf16(a, pdl, s, dev) : rows_ln_fp8_fp16(a, pdl, s, dev);
            return fns[a.norm == 1][a.gate != nullptr][dtype != 0](a, pdl, s, dev);
        }
        case LN_PATH_TOKENS: return ln_tokens_launch(a, dtype, pdl, s, dev);
        default: return ln_generic_launch(a, dtype, pdl, s, dev);
    }
}

cudaError_t launch_ln_modulate(const LnArgs &a, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    return launch_norm_scale_shift(a, dtype, pdl, s, dev);
}

}  // namespace adaln
