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
#include "ln_common.cuh"

namespace adaln {

// The contiguous-rows kernel moves every logical lane's vec4 chunk with one
// 8-byte access, so every row start of x, out, scale and shift must be
// 8-byte aligned.  Strides of size-1 dimensions are never used and are
// ignored.
bool ln_rows_ok(const LnArgs &a) {
    return ln_aligned(a.x, 8) && ln_aligned(a.out, 8) && ln_aligned(a.scale, 8) && ln_aligned(a.shift, 8) &&
           (a.N == 1 || ln_mult(a.sxN, 4)) &&
           (a.B == 1 || (ln_mult(a.sxB, 4) && ln_mult(a.s_scale_b, 4) && ln_mult(a.s_shift_b, 4)));
}

int ln_modulate_path(const LnArgs &a) {
    const int64_t ni = (a.D + 511) / 512;
    if (a.sxD == 1 && ni <= kRowsMaxNI && ln_rows_ok(a)) return LN_PATH_ROWS;
    // tokens contiguous: each d-row of 8 tokens is one 16-byte copy
    if (a.sxN == 1 && a.sxD != 1 && a.N > 1 && ni <= kTokensMaxNI && ln_aligned(a.x, 16) &&
        ln_mult(a.sxD, 8) && (a.B == 1 || (ln_mult(a.sxB, 8) && ln_mult(a.s_scale_b, 4) && ln_mult(a.s_shift_b, 4))) &&
        ln_aligned(a.out, 8) && ln_aligned(a.scale, 8) && ln_aligned(a.shift, 8))
        return LN_PATH_TOKENS;
    return LN_PATH_GENERIC;
}

cudaError_t launch_ln_modulate(const LnArgs &a, int dtype, bool pdl, cudaStream_t s,
                               const DeviceInfo &dev) {
    switch (ln_modulate_path(a)) {
        case LN_PATH_ROWS: return dtype == 0 ? ln_rows_bf16(a, pdl, s, dev) : ln_rows_fp16(a, pdl, s, dev);
        case LN_PATH_TOKENS: return ln_tokens_launch(a, dtype, pdl, s, dev);
        default: return ln_generic_launch(a, dtype, pdl, s, dev);
    }
}

// The fused kernel when the rows path takes these rows and y, r_out and the
// gate rows are 8-byte aligned with strides that keep them so; otherwise the
// gate-add kernel writes r and the LayerNorm reads it back (two launches).
bool residual_ln_fused_ok(const LnArgs &a, const void *y, const void *gate, int64_t s_gate_b, const void *r_out) {
    return ln_modulate_path(a) == LN_PATH_ROWS && ln_aligned(y, 8) && ln_aligned(r_out, 8) && ln_aligned(gate, 8) &&
           (a.B == 1 || ln_mult(s_gate_b, 4));
}

cudaError_t launch_residual_gate_ln_modulate(const LnArgs &a, const void *y, const void *gate, int64_t s_gate_b,
                                             void *r_out, int dtype, bool pdl, cudaStream_t s, const DeviceInfo &dev) {
    if (residual_ln_fused_ok(a, y, gate, s_gate_b, r_out))
        return dtype == 0 ? ln_rows_gate_bf16(a, y, gate, s_gate_b, r_out, pdl, s, dev)
                          : ln_rows_gate_fp16(a, y, gate, s_gate_b, r_out, pdl, s, dev);
    const GateArgs g{r_out, a.x, gate, s_gate_b, y, a.B, a.N, a.D};
    cudaError_t e = launch_residual_gate_add(g, dtype, pdl, s, dev);
    if (e != cudaSuccess) return e;
    LnArgs ln = a;
    ln.x = r_out;
    return launch_ln_modulate(ln, dtype, pdl, s, dev);
}

}  // namespace adaln
