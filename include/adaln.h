/*
 * adaln.h -- C ABI of the fused non-GEMM chains of a diffusion-transformer
 * block, for NVIDIA GB300 (sm_103a).
 *
 * The fused forms of eager PyTorch chains described on the SGLang Diffusion
 * "Fused Kernels" page and its pull-request pages:
 *
 *   adaln_ln_modulate          LayerNorm (no affine) + adaLN modulate
 *   adaln_qk_head_layernorm    per-head LayerNorm with affine on q and k
 *   adaln_residual_gate_add    x + gate * y
 *   adaln_bias_gelu_tanh       tanh-GELU of (x + bias)
 *   adaln_residual_gate_ln_modulate   x + gate * y, then LayerNorm + modulate
 *   adaln_norm_scale_shift     LayerNorm or RMSNorm + modulate, optional
 *                              residual gate, per-sample or per-token rows
 *   adaln_rmsnorm_scale_shift  RMSNorm (no affine) + modulate
 *   adaln_qk_rmsnorm           per-head RMSNorm with a weight on q and k
 *   adaln_temb_table_slices    table + temb as contiguous binary32 chunks
 *   adaln_ln_modulate_fp8      LayerNorm + adaLN modulate into static FP8
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Tensors are caller-owned device buffers of 16-bit storage values
 *    (bf16 or fp16, `adaln_dtype`); sizes and strides are in ELEMENTS.
 *  - Every operation is asynchronous on `stream` (a cudaStream_t; NULL is
 *    the legacy default stream) and never synchronises the host.
 *  - Arguments are validated entirely on the host before anything is
 *    launched.  On failure the call returns a non-zero `adaln_status`,
 *    launches nothing and leaves every buffer untouched.  A CUDA error at
 *    launch returns ADALN_E_CUDA (the CUDA error string is available from
 *    adaln_last_cuda_error()).  No C++ exception crosses this interface.
 *  - Arithmetic: binary32 with the storage rounding points of the eager
 *    chain; results are bit-identical for a given input on every launch
 *    geometry (a fixed reduction order, described per operation).
 *    NaN results are NaN; their payload bits are not specified.
 *  - adaln_can_* take the same arguments as the operation (minus the
 *    stream), run no CUDA call and return what the operation would return
 *    from validation (ADALN_OK when it would launch).
 *  - Thread safety: calls may be made from several host threads.
 *  - Memory: no call allocates device memory, except the one-time
 *    per-device GELU tables of adaln_bias_gelu_tanh (adaln_init).
 */
#ifndef ADALN_H
#define ADALN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum adaln_status {
    ADALN_OK = 0,
    ADALN_E_NULL = 1,    /* a required pointer is NULL */
    ADALN_E_DTYPE = 2,   /* dtype is not ADALN_BF16 / ADALN_FP16 */
    ADALN_E_SHAPE = 3,   /* a size is out of range (see each operation) */
    ADALN_E_ALIGN = 4,   /* a pointer is not aligned to the element size */
    ADALN_E_STRIDE = 5,  /* a stride is negative, above 2^46 elements, or not allowed */
    ADALN_E_VALUE = 6,   /* eps negative or not finite, or unknown flag bits */
    ADALN_E_OVERLAP = 7, /* an output overlaps an input in a way not allowed */
    ADALN_E_CUDA = 8     /* a CUDA runtime call failed */
} adaln_status;

typedef enum adaln_dtype {
    ADALN_BF16 = 0,
    ADALN_FP16 = 1,
    ADALN_FP32 = 2 /* IEEE binary32: only the inputs of adaln_temb_table_slices */
} adaln_dtype;

/* norm kinds of adaln_norm_scale_shift */
#define ADALN_NORM_LAYER 0 /* LayerNorm without affine */
#define ADALN_NORM_RMS 1   /* RMSNorm without affine */

/* flags */
#define ADALN_FLAG_PDL 1u /* launch with programmatic dependent launch: the
                             kernel may start while the previous kernel on
                             the stream finishes, and waits for it before
                             reading any input */

/* Human-readable name of a status code (static storage, never NULL). */
const char *adaln_status_str(int status);

/* Text of the last CUDA error seen by this library in the calling host
 * thread ("" if none). */
const char *adaln_last_cuda_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int adaln_version(void);

/* Diagnostic, not an operation of the pages.  Number of times, on the
 * current device since the library was loaded, that the transposed-view
 * ln_modulate kernel gave up waiting for its tensor-memory-accelerator
 * copies (a bounded wait; the affected tile is then left unwritten).  Stays
 * 0 unless the hardware fails to complete a copy.  Synchronous (a small
 * device-to-host read).  count: host pointer, written on ADALN_OK.
 * Returns ADALN_E_NULL or ADALN_E_CUDA on error. */
adaln_status adaln_tma_wait_timeouts(uint32_t *count);

/* One-time per-device set-up: queries the device and builds the two
 * 65536-entry GELU tables of adaln_bias_gelu_tanh (2 x 128 KiB of device
 * memory, owned by the library).  Synchronous.  Calling it is optional:
 * the first adaln_bias_gelu_tanh on a device does it too, which is not
 * allowed while the stream is being captured into a CUDA graph, so call
 * adaln_init first when capturing.  Idempotent. */
adaln_status adaln_init(int device);

/* Frees what adaln_init allocated, on every device.  Call only when no
 * operation of this library is in flight. */
adaln_status adaln_shutdown(void);

/* ------------------------------------------------------------------------
 * adaln_ln_modulate
 *   out[b, n, :] = LN(x[b, n, :]) * (1 + scale[b, :]) + shift[b, :]
 *
 * The fused "layernorm_modulate" of the Fused Kernels page (Normalization
 * table: affine-free LayerNorm + adaLN modulate, bit-exact contract), with
 * the tail-chunk generalisation to D % 4 == 0 of PR #34015 and the
 * per-sample (B, 1, D) scale / shift rows of PR #34008.
 *
 *   x      (B, N, D) with element strides (sxB, sxN, sxD): element (b,n,d)
 *          at x[b*sxB + n*sxN + d*sxD].  Contiguous (sxD == 1) and the
 *          transposed view of a contiguous (B, D, N) tensor (sxN == 1, as
 *          in Sana) have dedicated kernels; any other non-negative strides
 *          are accepted and take a slower general kernel.
 *   out    (B, N, D) contiguous.  May equal x only when x is contiguous
 *          (sxD == 1, sxN == D, sxB == N*D); otherwise must not overlap x.
 *   scale, shift  row b starts at scale + b*s_scale_b (resp. shift +
 *          b*s_shift_b) and is contiguous over D: the (B, 1, D) chunk views
 *          of an adaLN table (B, nmod, D) are (table + c*D, nmod*D).
 *   eps    finite, >= 0 (used as a binary32 value).
 *   Limits: B, N >= 1; 4 <= D <= 65536, D % 4 == 0.
 *
 * Numerics (fixed, independent of the launch geometry): 128 logical lanes;
 * lane l accumulates vec4 chunks j = i*128 + l (j < D/4) with the serial
 * Welford update mean' = fma(d, 1/(c+1), mean), m2' = fma(d, x - mean', m2)
 * (IEEE division); lanes are merged by Chan's pairwise combine in the
 * butterfly order 16, 8, 4, 2, 1, 64, 32; var = m2 / D; rstd = correctly
 * rounded 1/sqrt(var + eps); per element y = round(rstd*(x - mean)),
 * op = round(1 + scale), p = round(y*op), out = round(p + shift).
 * ---------------------------------------------------------------------- */
adaln_status adaln_ln_modulate(void *out, const void *x, int64_t B, int64_t N, int64_t D,
                               int64_t sxB, int64_t sxN, int64_t sxD,
                               const void *scale, int64_t s_scale_b,
                               const void *shift, int64_t s_shift_b,
                               float eps, int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_ln_modulate(const void *out, const void *x, int64_t B, int64_t N,
                                   int64_t D, int64_t sxB, int64_t sxN, int64_t sxD,
                                   const void *scale, int64_t s_scale_b,
                                   const void *shift, int64_t s_shift_b,
                                   float eps, int dtype, uint32_t flags);

/* Which kernel adaln_ln_modulate would launch for these arguments (no
 * launch): 0 = contiguous rows (sxD == 1, D <= 4096, 8-byte aligned rows),
 * 1 = contiguous tokens (sxN == 1, the transposed view; D <= 6144, 16-byte
 * aligned d-rows) through the cp.async tile kernel, 3 = the same view
 * through 16-token tensor-memory-accelerator tiles (D <= 5120 and a CUDA
 * driver present: this reads the current device's attributes once and
 * builds the tensor map on the host), 2 = general strides.  The numbers
 * are identical on every path.  Returns the negative adaln_status if the
 * arguments are invalid. */
int adaln_ln_modulate_variant(const void *out, const void *x, int64_t B, int64_t N,
                              int64_t D, int64_t sxB, int64_t sxN, int64_t sxD,
                              const void *scale, int64_t s_scale_b,
                              const void *shift, int64_t s_shift_b,
                              float eps, int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_qk_head_layernorm
 *   q_out[r, :] = LN(q[r, :]) * wq + bq,  k_out[r, :] = LN(k[r, :]) * wk + bk
 *
 * The "qk_head_layernorm" of the Fused Kernels page (per-head LayerNorm on
 * q / k, bit-exact) as used by GLM-Image (PR #34008): both tensors in ONE
 * launch.  q is (rows_q, Dh), k is (rows_k, Dh), both contiguous (rows =
 * B*N*H for a (B, N, H, Dh) tensor).  wq, bq, wk, bk are (Dh,) vectors
 * (the same pointers may be passed for q and k).  Outputs are contiguous;
 * q_out may equal q and k_out may equal k (in place); no other overlap.
 * rows_q or rows_k may be 0 (that tensor is skipped; its pointers may be
 * NULL), not both.
 *   Limits: 4 <= Dh <= 128, Dh % 4 == 0; eps finite, >= 0.
 * Numerics: as adaln_ln_modulate with 32 logical lanes (lane l holds
 * elements 4l..4l+3; butterfly 16, 8, 4, 2, 1), then
 * out = round(fma(w, rstd*(x - mean), b)) with one rounding.
 * ---------------------------------------------------------------------- */
adaln_status adaln_qk_head_layernorm(void *q_out, const void *q, int64_t rows_q,
                                     void *k_out, const void *k, int64_t rows_k, int64_t Dh,
                                     const void *wq, const void *bq,
                                     const void *wk, const void *bk,
                                     float eps, int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_qk_head_layernorm(const void *q_out, const void *q, int64_t rows_q,
                                         const void *k_out, const void *k, int64_t rows_k,
                                         int64_t Dh, const void *wq, const void *bq,
                                         const void *wk, const void *bk,
                                         float eps, int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_qk_rmsnorm
 *   q_out[r, :] = RMSNorm(q[r, :]) * wq,  k_out[r, :] = RMSNorm(k[r, :]) * wk
 *
 * The per-head QK RMSNorm of the Fused Kernels page (Normalization table:
 * qk_rmsnorm_native), q and k in one launch.  Shapes, layouts, limits,
 * aliasing and statuses as adaln_qk_head_layernorm without the biases
 * (rows of Dh contiguous values, 4 <= Dh <= 128, Dh % 4 == 0, 8-byte
 * aligned tensors; rows_q or rows_k may be 0 with its pointers NULL).
 * Numerics: 32 logical lanes, lane l holds elements 4l..4l+3 and sums
 * round(v * v) serially; lanes added in the butterfly order 16, 8, 4, 2, 1;
 * rstd = correctly rounded 1/sqrt(ss / Dh + eps); out = round(w * u) with
 * u = round(rstd * x), both products in binary32.
 * ---------------------------------------------------------------------- */
adaln_status adaln_qk_rmsnorm(void *q_out, const void *q, int64_t rows_q,
                              void *k_out, const void *k, int64_t rows_k, int64_t Dh,
                              const void *wq, const void *wk,
                              float eps, int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_qk_rmsnorm(const void *q_out, const void *q, int64_t rows_q,
                                  const void *k_out, const void *k, int64_t rows_k,
                                  int64_t Dh, const void *wq, const void *wk,
                                  float eps, int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_ln_modulate_fp8
 *   out[b, n, :] = e4m3(y / qscale),  y = LN(x) * (1 + scale) + shift
 *
 * The "flux2_layernorm_modulate_fp8_quant" of the Fused Kernels page
 * (Quantized layout producers table: LayerNorm plus adaLN modulation
 * directly into static FP8 output): adaln_ln_modulate followed by a static
 * per-tensor FP8 quantisation, the 16-bit y never written.
 *   out     (B, N, D) contiguous bytes, FP8 e4m3 (the finite-only variant:
 *           largest value 448, 0x7F / 0xFF NaN).
 *   qscale  DEVICE pointer to one binary32 scale (4-byte aligned), read by
 *           the kernel after earlier work on the stream; a positive finite
 *           value is expected (anything else gives what the IEEE division
 *           gives, then saturation).
 *   x, scale, shift, eps, dtype: as adaln_ln_modulate.  out overlaps no
 *           input (no in-place form: the element sizes differ).
 *   Kernels: the contiguous-rows kernel under its conditions, otherwise
 *   the general kernel (same bits); the transposed-view tile kernels do not
 *   write FP8.
 * Numerics: y exactly as adaln_ln_modulate stores it, then one IEEE
 * binary32 division by *qscale, round to nearest even to e4m3, saturating
 * at +-448 (infinities included); NaN stays NaN.
 * Cost: the rows kernel gets these codes from the product y * p alone when
 * a check over every significand of the storage type shows that, for a
 * multiplier p within 2 ulp of 1 / qscale, the product gives the division's
 * code for every 16-bit value.  Each CTA runs that check (about a
 * microsecond) only when the device's record of the last checked scale (one
 * per storage type, kept in device memory by the library) holds a
 * different scale, so calls that reuse a scale skip it; calls that
 * alternate scales on one device run it every time.  Scales that no
 * multiplier serves take an exact correction (a few operations more per
 * element).  The bits are the same in every case.
 * ---------------------------------------------------------------------- */
adaln_status adaln_ln_modulate_fp8(void *out, const void *qscale, const void *x,
                                  int64_t B, int64_t N, int64_t D,
                                  int64_t sxB, int64_t sxN, int64_t sxD,
                                  const void *scale, int64_t s_scale_b,
                                  const void *shift, int64_t s_shift_b,
                                  float eps, int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_ln_modulate_fp8(const void *out, const void *qscale, const void *x,
                                      int64_t B, int64_t N, int64_t D,
                                      int64_t sxB, int64_t sxN, int64_t sxD,
                                      const void *scale, int64_t s_scale_b,
                                      const void *shift, int64_t s_shift_b,
                                      float eps, int dtype, uint32_t flags);

/* Which kernel adaln_ln_modulate_fp8 would launch (codes of
 * adaln_ln_modulate_variant), or -status for invalid arguments. */
int adaln_ln_modulate_fp8_variant(const void *out, const void *qscale, const void *x,
                                  int64_t B, int64_t N, int64_t D,
                                  int64_t sxB, int64_t sxN, int64_t sxD,
                                  const void *scale, int64_t s_scale_b,
                                  const void *shift, int64_t s_shift_b,
                                  float eps, int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_temb_table_slices
 *   out_k[b, s, :] = table[k, :] + temb[b, s, k, :]      k = 0 .. K-1
 *
 * The "temb_table_slices" of the Fused Kernels page (adaLN modulation and
 * gating table and its note): the eager (scale_shift_table +
 * temb.float()).chunk(K, dim=2) as K slices, each contiguous, written in
 * one pass (no full binary32 sum materialised and no .contiguous() copies).
 *   out    binary32; slice k is the contiguous (B, S, D) block at
 *          out + k * s_out_k (floats); s_out_k >= B*S*D (ignored for K = 1).
 *   table  (K, D) contiguous, table_dtype ADALN_BF16 / ADALN_FP16 / ADALN_FP32.
 *   temb   (B, S, K, D) contiguous (S = 1 for one row per sample),
 *          temb_dtype likewise.
 *   Limits: B, S, K, D >= 1; K, D <= 65536.  out overlaps neither input.
 *   Pointers aligned to their element size; 8-wide accesses when D % 8 ==
 *   0, s_out_k % 8 == 0, out 32-byte and the inputs 8-element aligned,
 *   one element per access otherwise (same bits).
 * Numerics: one IEEE binary32 addition of the exactly promoted operands.
 * Returns ADALN_E_DTYPE for a dtype outside the three, ADALN_E_STRIDE for
 * s_out_k < B*S*D, and the common statuses.
 * ---------------------------------------------------------------------- */
adaln_status adaln_temb_table_slices(void *out, int64_t s_out_k, const void *table, int table_dtype,
                                    const void *temb, int temb_dtype,
                                    int64_t B, int64_t S, int64_t K, int64_t D,
                                    uint32_t flags, void *stream);

adaln_status adaln_can_temb_table_slices(const void *out, int64_t s_out_k, const void *table,
                                        int table_dtype, const void *temb, int temb_dtype,
                                        int64_t B, int64_t S, int64_t K, int64_t D,
                                        uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_residual_gate_add
 *   out[b, n, d] = x[b, n, d] + gate[b, d] * y[b, n, d]
 *
 * The "residual_gate_add" of the Fused Kernels page (adaLN modulation and
 * gating table: residual + gate * update, bit-exact), GLM-Image's ff-gate
 * (PR #34008).  x, y, out contiguous (B, N, D); gate row b at
 * gate + b*s_gate_b, contiguous over D (a (B, 1, D) tensor has
 * s_gate_b = D).  out may equal x or y; no other overlap.
 *   Limits: B, N >= 1; D >= 1.
 * Numerics: out = round(x + round(gate * y)) (two storage roundings, no
 * fused multiply-add).
 * ---------------------------------------------------------------------- */
adaln_status adaln_residual_gate_add(void *out, const void *x, const void *gate,
                                     int64_t s_gate_b, const void *y,
                                     int64_t B, int64_t N, int64_t D,
                                     int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_residual_gate_add(const void *out, const void *x, const void *gate,
                                         int64_t s_gate_b, const void *y,
                                         int64_t B, int64_t N, int64_t D,
                                         int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_residual_gate_ln_modulate
 *   r_out[b, n, :] = x[b, n, :] + gate[b, :] * y[b, n, :]
 *   out[b, n, :]   = LN(r_out[b, n, :]) * (1 + scale[b, :]) + shift[b, :]
 *
 * The "scale_residual_norm_scale_shift" of the Fused Kernels page (Kernel
 * inventory, Normalization table: the norm + scale/shift chain together
 * with the preceding residual + gate * update), with the LayerNorm of
 * adaln_ln_modulate: the residual gate-add and the following LN+modulate of
 * a DiT block in one pass, x and y read once, r and out written once.
 *   x, y, r_out, out contiguous (B, N, D); gate, scale, shift rows at
 *   ptr + b * stride, contiguous over D (stride 0 broadcasts one row).
 *   r_out may equal x or y (an in-place residual update); out overlaps none
 *   of the others.
 *   Limits: those of adaln_residual_gate_add and adaln_ln_modulate (D % 4
 *   == 0, eps finite and >= 0).  One launch: the contiguous-rows kernel when
 *   D <= 4096, the rows are 8-byte aligned and the gate rows are 8-byte
 *   aligned with s_gate_b % 4 == 0; otherwise the general kernel (same
 *   bits).  This is adaln_norm_scale_shift with ADALN_NORM_LAYER, one gate,
 *   scale and shift row per sample.
 * Numerics: r_out = round(x + round(gate * y)); out is adaln_ln_modulate of
 * r_out as stored (bit for bit the two calls in sequence).
 * Returns the statuses of the two calls it combines; ADALN_E_OVERLAP also
 * when out overlaps x, y, r_out or the gate rows, or r_out overlaps the
 * scale or shift rows.
 * ---------------------------------------------------------------------- */
adaln_status adaln_residual_gate_ln_modulate(void *r_out, void *out, const void *x,
                                             const void *gate, int64_t s_gate_b,
                                             const void *y, int64_t B, int64_t N, int64_t D,
                                             const void *scale, int64_t s_scale_b,
                                             const void *shift, int64_t s_shift_b,
                                             float eps, int dtype, uint32_t flags,
                                             void *stream);

/* ------------------------------------------------------------------------
 * adaln_norm_scale_shift
 *   v[b, n, :]     = x[b, n, :]                                  (gate NULL)
 *   v[b, n, :]     = x[b, n, :] + gate[b, n, :] * y[b, n, :]     (otherwise;
 *                                                   stored to r_out)
 *   out[b, n, :]   = norm(v[b, n, :]) * (1 + scale[b, n, :]) + shift[b, n, :]
 *
 * The norm + scale/shift chains of the Fused Kernels page (Normalization
 * table: layernorm_modulate, rmsnorm_scale_shift and, with a gate,
 * scale_residual_norm_scale_shift) with the broadcast modes of its
 * request-gated fusion table: per-token [B, S, 1] gates and per-token
 * modulation rows read through strided [B, S, 6D] chunk views.
 *   norm   ADALN_NORM_LAYER (affine-free LayerNorm, the statistics of
 *          adaln_ln_modulate) or ADALN_NORM_RMS (affine-free RMSNorm).
 *   x      (B, N, D), element (b, n, d) at x[b*sxB + n*sxN + d*sxD]; with a
 *          gate x must be contiguous (sxD == 1, sxN == D, sxB == N*D).
 *   gate   NULL, or element (b, n, d) at gate[b*s_gate_b + n*s_gate_n +
 *          d*s_gate_d] with s_gate_d 1 (a row) or 0 (one value per token,
 *          a [B, S, 1] gate); s_gate_n == 0 broadcasts one row per sample.
 *   y, r_out  with a gate: (B, N, D) contiguous; r_out may equal x or y (an
 *          in-place residual update), out overlaps none of x, y, r_out and
 *          the gate.  Ignored (may be NULL) without a gate.
 *   scale, shift  element (b, n, d) at scale[b*s_scale_b + n*s_scale_n + d]
 *          (contiguous over d): s_scale_n == 0 gives the per-sample (B, 1, D)
 *          rows; the chunk c of a per-token (B, N, nmod*D) table is
 *          (table + c*D, N*nmod*D, nmod*D).
 *   out    (B, N, D) contiguous; may equal x only without a gate and when x
 *          is contiguous.  r_out and out overlap no scale / shift element.
 *   Limits: B, N >= 1; 4 <= D <= 65536, D % 4 == 0; eps finite and >= 0.
 *   Kernels: the contiguous-rows kernel when x is contiguous over d,
 *   D <= 4096 and the rows (and strides) keep 8-byte alignment; the
 *   transposed-view tile kernels for the LayerNorm with per-sample rows and
 *   no gate; otherwise a general kernel.  Every kernel gives the same bits.
 * Numerics: with a gate v = round(x + round(gate * y)) as stored in r_out.
 *   LayerNorm: the Welford / Chan DAG of adaln_ln_modulate.  RMSNorm: the
 *   same 128 logical lanes and chunk order, each lane accumulating
 *   s = round(s + round(v * v)), lanes added in the butterfly order 16, 8,
 *   4, 2, 1, 64, 32, ms = s / D, rstd = correctly rounded 1/sqrt(ms + eps),
 *   mean taken as 0.  Then per element y = round(rstd * (v - mean)),
 *   op = round(1 + scale), p = round(y * op), out = round(p + shift).
 * Returns ADALN_E_VALUE for an unknown norm, ADALN_E_NULL for a gate
 * without y or r_out, ADALN_E_STRIDE for a gate with non-contiguous x or
 * s_gate_d other than 0 / 1, and the statuses of adaln_ln_modulate.
 * ---------------------------------------------------------------------- */
adaln_status adaln_norm_scale_shift(int norm, void *r_out, void *out, const void *x,
                                    int64_t B, int64_t N, int64_t D,
                                    int64_t sxB, int64_t sxN, int64_t sxD,
                                    const void *gate, int64_t s_gate_b, int64_t s_gate_n,
                                    int64_t s_gate_d, const void *y,
                                    const void *scale, int64_t s_scale_b, int64_t s_scale_n,
                                    const void *shift, int64_t s_shift_b, int64_t s_shift_n,
                                    float eps, int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_norm_scale_shift(int norm, const void *r_out, const void *out,
                                        const void *x, int64_t B, int64_t N, int64_t D,
                                        int64_t sxB, int64_t sxN, int64_t sxD,
                                        const void *gate, int64_t s_gate_b, int64_t s_gate_n,
                                        int64_t s_gate_d, const void *y,
                                        const void *scale, int64_t s_scale_b, int64_t s_scale_n,
                                        const void *shift, int64_t s_shift_b, int64_t s_shift_n,
                                        float eps, int dtype, uint32_t flags);

/* Which kernel adaln_norm_scale_shift would launch, with the codes of
 * adaln_ln_modulate_variant, or -status when the arguments are invalid. */
int adaln_norm_scale_shift_variant(int norm, const void *r_out, const void *out,
                                   const void *x, int64_t B, int64_t N, int64_t D,
                                   int64_t sxB, int64_t sxN, int64_t sxD,
                                   const void *gate, int64_t s_gate_b, int64_t s_gate_n,
                                   int64_t s_gate_d, const void *y,
                                   const void *scale, int64_t s_scale_b, int64_t s_scale_n,
                                   const void *shift, int64_t s_shift_b, int64_t s_shift_n,
                                   float eps, int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_rmsnorm_scale_shift
 *   out[b, n, :] = RMSNorm(x[b, n, :]) * (1 + scale[b, n, :]) + shift[b, n, :]
 *
 * The "rmsnorm_scale_shift" of the Fused Kernels page (Normalization table:
 * RMSNorm + `* (1 + scale) + shift`, bit-exact, replacing four kernels):
 * adaln_norm_scale_shift with ADALN_NORM_RMS and no gate; same arguments,
 * limits, numerics and statuses.
 * ---------------------------------------------------------------------- */
adaln_status adaln_rmsnorm_scale_shift(void *out, const void *x, int64_t B, int64_t N, int64_t D,
                                       int64_t sxB, int64_t sxN, int64_t sxD,
                                       const void *scale, int64_t s_scale_b, int64_t s_scale_n,
                                       const void *shift, int64_t s_shift_b, int64_t s_shift_n,
                                       float eps, int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_rmsnorm_scale_shift(const void *out, const void *x, int64_t B, int64_t N,
                                           int64_t D, int64_t sxB, int64_t sxN, int64_t sxD,
                                           const void *scale, int64_t s_scale_b, int64_t s_scale_n,
                                           const void *shift, int64_t s_shift_b, int64_t s_shift_n,
                                           float eps, int dtype, uint32_t flags);

adaln_status adaln_can_residual_gate_ln_modulate(const void *r_out, const void *out,
                                                 const void *x, const void *gate,
                                                 int64_t s_gate_b, const void *y,
                                                 int64_t B, int64_t N, int64_t D,
                                                 const void *scale, int64_t s_scale_b,
                                                 const void *shift, int64_t s_shift_b,
                                                 float eps, int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_bias_gelu_tanh
 *   out[r, c] = gelu_tanh(round(x[r, c] + bias[c]))
 *
 * The bias + tanh-GELU epilogue of the Wan2.2 FFN (PR #37075, "功能与动机"
 * and the bias_gelu_tanh kernel): fp32 add, rounded back to the storage
 * type BEFORE the activation, then tanh-GELU, rounded again.  x, out
 * contiguous (rows, width); bias (width,).  out may equal x.
 *   Limits: rows >= 1; width >= 1.
 * Numerics: gelu_tanh(v) is the binary32 value nearest to the exact
 * 0.5*v*(1 + tanh(sqrt(2/pi)*(v + 0.044715*v^3))), then rounded to the
 * storage type; it is read from a 65536-entry table per dtype (built once
 * per device, see adaln_init), exact for every input.
 * ---------------------------------------------------------------------- */
adaln_status adaln_bias_gelu_tanh(void *out, const void *x, const void *bias,
                                  int64_t rows, int64_t width,
                                  int dtype, uint32_t flags, void *stream);

adaln_status adaln_can_bias_gelu_tanh(const void *out, const void *x, const void *bias,
                                      int64_t rows, int64_t width,
                                      int dtype, uint32_t flags);

/* ------------------------------------------------------------------------
 * adaln_copy_reference
 *   Copies `bytes` bytes from src to dst on `stream` with a kernel built like
 *   the ops' streaming kernels (32-byte accesses that bypass L1, a persistent
 *   grid sized from the SM count, ADALN_FLAG_PDL as for the ops).  The pages
 *   have no counterpart: it is the same-byte yardstick that measurements put
 *   beside each op (an op that moves R + W bytes is compared with a copy of
 *   (R + W) / 2 bytes).
 *   dst, src: device pointers, 32-byte aligned (else ADALN_E_ALIGN), not
 *   overlapping (else ADALN_E_OVERLAP); bytes in [1, 2^46] (else
 *   ADALN_E_SHAPE); flags 0 or ADALN_FLAG_PDL (else ADALN_E_VALUE).
 *   Asynchronous; returns ADALN_E_CUDA if the launch fails.
 * ---------------------------------------------------------------------- */
adaln_status adaln_copy_reference(void *dst, const void *src, int64_t bytes, uint32_t flags, void *stream);

/* ------------------------------------------------------------------------
 * adaln_bias_gelu_tanh_noalloc
 *   The same operation, arguments, limits and results (bit for bit) as
 *   adaln_bias_gelu_tanh, for callers that cannot let a library allocate
 *   device memory.  The paper has no counterpart: this entry point exists
 *   for the way some programs manage memory, not for the method.
 *
 *   Who needs it: a process whose memory pool or arena owns the whole device
 *   (a server that plans every byte of HBM up front), code that must not
 *   hit the implicit device synchronisation of cudaMalloc / cudaFree, or a
 *   host program that forbids allocations after start-up.
 *   adaln_bias_gelu_tanh allocates its lookup tables with cudaMalloc on
 *   first use; this variant keeps them in a fixed array that is part of the
 *   library's device image and calls no cudaMalloc, cudaFree or other
 *   allocating routine.  The caller still allocates and owns x, bias, out.
 *
 *   Memory held: 256 KiB (one 65536-entry table per storage type) on every
 *   GPU that loads the library, until the process exits.  The array holds
 *   lookup tables, not data of the call: its size does not depend on rows
 *   or width, both storage types' tables always fit, and the limits on
 *   rows and width are those of adaln_bias_gelu_tanh.
 *
 *   Set-up: the first call on a device for a storage type (made with that
 *   device current) looks up the array's device address and fills that
 *   storage type's table on `stream`, then waits for the stream to finish
 *   (so it runs after work already queued on `stream`).  Make that first
 *   call before capturing `stream` into a CUDA graph: a first call on a
 *   stream that is being captured returns ADALN_E_CUDA, with a message from
 *   adaln_last_cuda_error(), and leaves the capture untouched.  The
 *   table is written only by that first call; later calls only read the
 *   shared array, and nothing in it has to start at zero.  A later call
 *   that overlaps that first call's table build on another stream would
 *   race with it, and a call after cudaDeviceReset would use an array whose
 *   contents were lost; neither is detected.
 * ---------------------------------------------------------------------- */
adaln_status adaln_bias_gelu_tanh_noalloc(void *out, const void *x, const void *bias,
                                          int64_t rows, int64_t width,
                                          int dtype, uint32_t flags, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ADALN_H */
