/*
 * CPU oracle for the fused non-GEMM chains of a diffusion-transformer block.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The CUDA
 * library never calls, links or includes anything here, and this file shares
 * no code, header, table or constant generator with it.
 *
 * Plain, slow, scalar C.  Every floating-point step is one IEEE binary32
 * operation rounded to nearest-even (compiled with -ffp-contract=off and no
 * fast-math, so `a * b + c` is never fused); `fmaf` is the single-rounding
 * fused multiply-add of C99.  Storage values are 16-bit patterns: bf16
 * (dtype 0) or fp16 (dtype 1).
 *
 * Sources (SGLang Diffusion "Fused Kernels" page and its pull-request pages):
 *  - LayerNorm + adaLN modulate: "Fused Kernels", Normalization table
 *    (layernorm_modulate) and "Numerical contracts and quality tiers"
 *    (serial Welford, guarded reciprocal, warp-fold tree); PR #34015
 *    "实现拆解" 1 (pass 1 over vec4 chunks, (D+511)//512 iterations, tail lanes
 *    whose vec index reaches D/4 skip; pass 2 rounding points of the
 *    modulate); PR #34008 "关键源码片段" (_welford_push update order).
 *  - qk_head_layernorm: "Fused Kernels", Normalization table; PR #34008
 *    "实现拆解" 1 (per-head LayerNorm on q and k in one kernel).
 *  - residual_gate_add: "Fused Kernels", adaLN modulation and gating table.
 *  - rmsnorm_scale_shift, scale_residual_norm_scale_shift, qk_rmsnorm_native:
 *    "Fused Kernels", Normalization table (RMSNorm + `* (1 + scale) + shift`;
 *    the same after `residual + gate * update`; per-head QK RMSNorm), the
 *    request-gated fusion table (per-token [B, S, 1] gate, strided
 *    [B, S, 6D] chunk views of the modulation rows) and "Numerical contracts
 *    and quality tiers" (the RMSNorm statistics are folded by a butterfly).
 *  - bias_gelu_tanh: PR #37075 "功能与动机" and "关键源码片段" (fp32 add,
 *    round to the storage type, then tanh-GELU, round again).
 *  - temb_table_slices: "Fused Kernels", adaLN modulation and gating table
 *    and its note on the op ((scale_shift_table + temb.float()).chunk(6)
 *    into six contiguous slices in one pass).
 *  - static FP8 output of LN + modulate: "Fused Kernels", Quantized layout
 *    producers table (flux2_layernorm_modulate_fp8_quant: LayerNorm plus
 *    adaLN modulation directly into static FP8 output).
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes): the reciprocal in the Welford push and every division are IEEE
 * round-to-nearest (not the pages' hardware-approximate reciprocal); rstd is
 * the correctly rounded 1/sqrt; var = m2 / D; the combine is Chan's pairwise
 * formula with a guarded coefficient; the fold is a butterfly over logical
 * lane bits in the order 16, 8, 4, 2, 1 then 64, 32; GELU's fp32 value is the
 * correctly rounded exact tanh-GELU.  RMSNorm: each lane sums x*x over its
 * chunks with the square and the sum rounded separately (no fused
 * multiply-add), the lanes are folded by the same butterfly with plain
 * additions, ms = ss / D, rstd = rsqrt_cr(ms + eps), and the normalised value
 * is round16(rstd * x), the LayerNorm's formula with mean 0.  The per-head
 * QK RMSNorm scales by its weight in binary32 and rounds once to storage.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* binary32 <-> 16-bit storage                                          */
/* ------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

/* bf16 -> f32: exact (bf16 is the top half of a binary32). */
static float bf16_to_f32(uint16_t h) { return f32_from_bits((uint32_t)h << 16); }

/* fp16 -> f32: exact, from the binary16 definition. */
static float f16_to_f32(uint16_t h) {
    uint32_t sign = (uint32_t)(h & 0x8000) << 16;
    uint32_t e = (h >> 10) & 0x1f, m = h & 0x3ff;
    if (e == 0x1f) return f32_from_bits(sign | 0x7f800000u | (m << 13));
    if (e == 0) {
        /* zero or subnormal: m * 2^-24, exact in binary32 */
        float v = (float)m * 0x1.0p-24f;
        return sign ? -v : v;
    }
    return f32_from_bits(sign | ((e + 112u) << 23) | (m << 13));
}

/* f32 -> bf16, round to nearest even; NaN -> canonical 0x7FC0. */
static uint16_t f32_to_bf16(float f) {
    uint32_t u = f32_bits(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0;
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7fffu + lsb) >> 16);
}

/* f32 -> fp16, round to nearest even, subnormals kept, overflow -> inf,
 * NaN -> canonical 0x7E00. */
static uint16_t f32_to_f16(float f) {
    uint32_t u = f32_bits(f);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t a = u & 0x7fffffffu;
    if (a > 0x7f800000u) return 0x7e00;
    if (a >= 0x477ff000u) return sign | 0x7c00; /* |f| >= 65520: rounds to inf */
    if (a >= 0x38800000u) {                     /* |f| >= 2^-14: normal result */
        uint32_t r = a - 0x38000000u;           /* rebias exponent 127 -> 15 */
        uint32_t lsb = (r >> 13) & 1u;
        return sign | (uint16_t)((r + 0xfffu + lsb) >> 13);
    }
    uint32_t E = a >> 23;                       /* subnormal result or zero */
    if (E < 102) return sign;                   /* |f| <= 2^-25 ... rounds to 0 */
    uint32_t m = (a & 0x7fffffu) | 0x800000u;   /* |f| = m * 2^(E-150) */
    uint32_t shift = 126 - E;                   /* result = RNE(m / 2^shift) */
    uint32_t q = m >> shift, rem = m & ((1u << shift) - 1u), half = 1u << (shift - 1);
    if (rem > half || (rem == half && (q & 1u))) ++q;
    return sign | (uint16_t)q;
}

static float load16(uint16_t h, int dtype) { return dtype ? f16_to_f32(h) : bf16_to_f32(h); }
static uint16_t store16(float f, int dtype) { return dtype ? f32_to_f16(f) : f32_to_bf16(f); }
/* one storage rounding, kept as binary32 (exact round trip) */
static float round16(float f, int dtype) { return load16(store16(f, dtype), dtype); }

/* ------------------------------------------------------------------ */
/* correctly rounded 1/sqrt(x) in binary32                              */
/* ------------------------------------------------------------------ */

/* x = M * 2^e exactly (M integer, 0 < M < 2^24), for finite x > 0 */
static void split_f32(float x, uint64_t *M, int *e) {
    uint32_t u = f32_bits(x), E = (u >> 23) & 0xff, m = u & 0x7fffffu;
    if (E == 0) { *M = m; *e = -149; }
    else { *M = m | 0x800000u; *e = (int)E - 150; }
}

/* sign of (mid^2 * x - 1), mid = (a + b) / 2, a, b, x finite positive floats */
static int mid_sq_times_x_vs_one(float a, float b, float x) {
    uint64_t A, Bm, X; int ea, eb, ex;
    split_f32(a, &A, &ea); split_f32(b, &Bm, &eb); split_f32(x, &X, &ex);
    int e = ea < eb ? ea : eb;
    uint64_t S = (A << (ea - e)) + (Bm << (eb - e));    /* a + b = S * 2^e, S < 2^26 */
    /* mid^2 * x = S^2 * X * 2^(2(e-1) + ex) */
    unsigned __int128 P = (unsigned __int128)(S * S) * X; /* < 2^76 */
    int k = 2 * (e - 1) + ex;
    if (k >= 0) return (P == 1 && k == 0) ? 0 : 1;
    if (-k >= 127) return -1;
    unsigned __int128 one = (unsigned __int128)1 << (-k);
    return P > one ? 1 : (P < one ? -1 : 0);
}

float oracle_rsqrt_cr(float x) {
    if (isnan(x) || x < 0.0f) return NAN;
    if (x == 0.0f) return signbit(x) ? -INFINITY : INFINITY;
    if (isinf(x)) return 0.0f;
    float r = (float)(1.0 / sqrt((double)x));
    /* r is correct iff lo_mid < 1/sqrt(x) < hi_mid, i.e.
     * lo_mid^2 * x < 1 < hi_mid^2 * x (no exact ties exist). */
    for (int it = 0; it < 4; ++it) {
        float up = nextafterf(r, INFINITY), dn = nextafterf(r, 0.0f);
        if (mid_sq_times_x_vs_one(r, up, x) <= 0) { r = up; continue; }
        if (mid_sq_times_x_vs_one(dn, r, x) >= 0) { r = dn; continue; }
        return r;
    }
    fprintf(stderr, "oracle_rsqrt_cr: did not settle for %a\n", (double)x);
    abort();
}

/* ------------------------------------------------------------------ */
/* Welford / Chan statistics on the canonical lane DAG                  */
/* ------------------------------------------------------------------ */

typedef struct { float mean, m2, cnt; } wstate;

/* one serial Welford step: mean' = fma(d, 1/(cnt+1), mean),
 * m2' = fma(d, v - mean', m2), with d = v - mean and an IEEE division. */
static void welford_push(wstate *s, float v) {
    float d = v - s->mean;
    float c1 = s->cnt + 1.0f;
    float r = 1.0f / c1;
    float mean = fmaf(d, r, s->mean);
    float t = v - mean;
    s->m2 = fmaf(d, t, s->m2);
    s->mean = mean;
    s->cnt = c1;
}

/* Chan's pairwise combine of a (lower lane) and b (upper lane):
 * n = na + nb, coef = nb / n (0 when n == 0), delta = mb - ma,
 * mean = fma(delta, coef, ma), m2 = fma(delta^2 * na, coef, m2a + m2b). */
static wstate chan_combine(wstate a, wstate b) {
    wstate o;
    float n = a.cnt + b.cnt;
    float coef = (n == 0.0f) ? 0.0f : b.cnt / n;
    float delta = b.mean - a.mean;
    o.mean = fmaf(delta, coef, a.mean);
    float dd = delta * delta;
    float dda = dd * a.cnt;
    float m2s = a.m2 + b.m2;
    o.m2 = fmaf(dda, coef, m2s);
    o.cnt = n;
    return o;
}

/* Statistics of one row of D values (already in binary32) over L logical
 * lanes (128 for ln_modulate, 32 for qk_head_layernorm).
 * Lane l owns vec4 chunks j = i*L + l, j < D/4, pushed in increasing i and
 * element order 4j..4j+3; lanes past the tail push nothing.  Then a
 * butterfly: at each stage offset o every lane l becomes
 * combine(state[l & ~o], state[l | o]).  Offsets 16, 8, 4, 2, 1 (inside a
 * group of 32 lanes) and then, for L = 128, 64, 32 (across groups). */
static const int order128[7] = {16, 8, 4, 2, 1, 64, 32};
static const int order32[5] = {16, 8, 4, 2, 1};

static void row_stats(const float *x, int64_t D, int L, float *mean, float *m2) {
    wstate st[128], nx[128];
    int64_t nvec = D / 4;
    for (int l = 0; l < L; ++l) {
        st[l].mean = 0.0f; st[l].m2 = 0.0f; st[l].cnt = 0.0f;
        for (int64_t j = l; j < nvec; j += L)
            for (int e = 0; e < 4; ++e) welford_push(&st[l], x[4 * j + e]);
    }
    const int *order = (L == 128) ? order128 : order32;
    int stages = (L == 128) ? 7 : 5;
    for (int s = 0; s < stages; ++s) {
        int o = order[s];
        for (int l = 0; l < L; ++l) nx[l] = chan_combine(st[l & ~o], st[l | o]);
        memcpy(st, nx, sizeof(wstate) * (size_t)L);
    }
    *mean = st[0].mean;
    *m2 = st[0].m2;
}

/* var = m2 / D; rstd = rsqrt_cr(var + eps) */
static float stats_rstd(float m2, int64_t D, float eps) {
    float var = m2 / (float)D;
    return oracle_rsqrt_cr(var + eps);
}

/* Sum of squares of one row on L logical lanes, for RMSNorm.  Lane l owns
 * the same vec4 chunks as in row_stats and accumulates s = s + x*x over
 * them in increasing chunk and element order (the square rounded to
 * binary32, then the sum: two roundings); lanes past the tail add nothing.
 * Then the butterfly of row_stats with s[l] = s[l & ~o] + s[l | o]. */
static float row_sumsq(const float *x, int64_t D, int L) {
    float st[128], nx[128];
    int64_t nvec = D / 4;
    for (int l = 0; l < L; ++l) {
        st[l] = 0.0f;
        for (int64_t j = l; j < nvec; j += L)
            for (int e = 0; e < 4; ++e) {
                float sq = x[4 * j + e] * x[4 * j + e];
                st[l] = st[l] + sq;
            }
    }
    const int *order = (L == 128) ? order128 : order32;
    int stages = (L == 128) ? 7 : 5;
    for (int s = 0; s < stages; ++s) {
        int o = order[s];
        for (int l = 0; l < L; ++l) nx[l] = st[l & ~o] + st[l | o];
        memcpy(st, nx, sizeof(float) * (size_t)L);
    }
    return st[0];
}

/* ms = ss / D; rstd = rsqrt_cr(ms + eps) */
static float rms_rstd(float ss, int64_t D, float eps) {
    float ms = ss / (float)D;
    return oracle_rsqrt_cr(ms + eps);
}

/* r = round16(x + round16(gate * y)): the residual gate-add of one element */
static float gate_add(float xv, uint16_t g, uint16_t yv, int dtype) {
    float gy = round16(load16(g, dtype) * load16(yv, dtype), dtype);
    return round16(xv + gy, dtype);
}

/* ------------------------------------------------------------------ */
/* norm + adaLN modulate (LayerNorm or RMSNorm, optional residual gate)  */
/* ------------------------------------------------------------------ */

/*
 * out[b, n, :] = modulate(norm(v[b, n, :])) for rows r = b*N + n in
 * [row_begin, row_end), where
 *   v = x                                   when gate is NULL,
 *   v = round16(x + round16(gate * y))      otherwise (the residual
 *                                           gate-add; r_out, if not NULL,
 *                                           receives v),
 * x element (b, n, d) at x[b*sxB + n*sxN + d*sxD], y contiguous (B, N, D),
 * gate (b, n, d) at gate[b*s_gate_b + n*s_gate_n + d*s_gate_d] (a per-token
 * [B, S, 1] gate has s_gate_d = 0), scale / shift (b, n, d) at
 * scale[b*s_scale_b + n*s_scale_n + d] (per-sample rows: s_scale_n = 0;
 * per-token rows, e.g. chunks of a [B, S, 6D] table: s_scale_n = 6D).
 * norm 0 is LayerNorm without affine (row_stats, stats_rstd); norm 1 is
 * RMSNorm without affine (row_sumsq, rms_rstd, mean 0).  Per element:
 *   y   = round16(rstd * (v - mean))
 *   op  = round16(1 + scale)
 *   p   = round16(y * op)
 *   out = round16(p + shift)
 * Row r goes to out + (r - row_begin) * D (and r_out likewise).  Optional
 * row_mean / row_rstd, indexed the same way, receive the statistics.
 * Returns 0, or -1 for D not a positive multiple of 4 or a bad norm.
 */
int oracle_norm_scale_shift(uint16_t *r_out, uint16_t *out, int norm,
                            const uint16_t *x, int64_t B, int64_t N, int64_t D,
                            int64_t sxB, int64_t sxN, int64_t sxD,
                            const uint16_t *gate, int64_t s_gate_b, int64_t s_gate_n,
                            int64_t s_gate_d, const uint16_t *y,
                            const uint16_t *scale, int64_t s_scale_b, int64_t s_scale_n,
                            const uint16_t *shift, int64_t s_shift_b, int64_t s_shift_n,
                            float eps, int dtype, int64_t row_begin, int64_t row_end,
                            float *row_mean, float *row_rstd) {
    if (D <= 0 || D % 4 || (norm != 0 && norm != 1)) return -1;
    float *v = (float *)malloc(sizeof(float) * (size_t)D);
    if (!v) return -2;
    for (int64_t r = row_begin; r < row_end && r < B * N; ++r) {
        int64_t b = r / N, n = r % N;
        const uint16_t *xr = x + b * sxB + n * sxN;
        for (int64_t d = 0; d < D; ++d) v[d] = load16(xr[d * sxD], dtype);
        if (gate) {
            const uint16_t *g = gate + b * s_gate_b + n * s_gate_n;
            for (int64_t d = 0; d < D; ++d) v[d] = gate_add(v[d], g[d * s_gate_d], y[r * D + d], dtype);
            if (r_out)
                for (int64_t d = 0; d < D; ++d) r_out[(r - row_begin) * D + d] = store16(v[d], dtype);
        }
        float mean, rstd;
        if (norm == 0) {
            float m2;
            row_stats(v, D, 128, &mean, &m2);
            rstd = stats_rstd(m2, D, eps);
        } else {
            mean = 0.0f;
            rstd = rms_rstd(row_sumsq(v, D, 128), D, eps);
        }
        if (row_mean) row_mean[r - row_begin] = mean;
        if (row_rstd) row_rstd[r - row_begin] = rstd;
        const uint16_t *sc = scale + b * s_scale_b + n * s_scale_n, *sh = shift + b * s_shift_b + n * s_shift_n;
        uint16_t *o = out + (r - row_begin) * D;
        for (int64_t d = 0; d < D; ++d) {
            float centered = v[d] - mean;
            float y = round16(rstd * centered, dtype);
            float op = round16(1.0f + load16(sc[d], dtype), dtype);
            float p = round16(y * op, dtype);
            o[d] = store16(p + load16(sh[d], dtype), dtype);
        }
    }
    free(v);
    return 0;
}

/* ln_modulate: LayerNorm (no affine) + adaLN modulate with one scale /
 * shift row per sample (row b at scale + b*s_scale_b); out contiguous
 * (B, N, D).  The norm 0, gate-free case of oracle_norm_scale_shift. */
int oracle_ln_modulate(uint16_t *out, const uint16_t *x, int64_t B, int64_t N, int64_t D,
                       int64_t sxB, int64_t sxN, int64_t sxD,
                       const uint16_t *scale, int64_t s_scale_b,
                       const uint16_t *shift, int64_t s_shift_b,
                       float eps, int dtype, int64_t row_begin, int64_t row_end,
                       float *row_mean, float *row_rstd) {
    return oracle_norm_scale_shift(NULL, out, 0, x, B, N, D, sxB, sxN, sxD, NULL, 0, 0, 0, NULL,
                                   scale, s_scale_b, 0, shift, s_shift_b, 0, eps, dtype,
                                   row_begin, row_end, row_mean, row_rstd);
}

/* ------------------------------------------------------------------ */
/* qk_head_layernorm                                                    */
/* ------------------------------------------------------------------ */

/* One tensor: rows of Dh contiguous values, LayerNorm with affine
 * out = round16(fma(w, rstd * (x - mean), b)) on 32 logical lanes.
 * Rows [row_begin, row_end); row r goes to out + (r - row_begin) * Dh.
 * Returns -1 unless 0 < Dh <= 128 and Dh % 4 == 0. */
int oracle_qk_head_layernorm(uint16_t *out, const uint16_t *in, int64_t rows, int64_t Dh,
                             const uint16_t *w, const uint16_t *bias, float eps, int dtype,
                             int64_t row_begin, int64_t row_end) {
    if (Dh <= 0 || Dh > 128 || Dh % 4) return -1;
    float v[128];
    for (int64_t r = row_begin; r < row_end && r < rows; ++r) {
        const uint16_t *xr = in + r * Dh;
        for (int64_t d = 0; d < Dh; ++d) v[d] = load16(xr[d], dtype);
        float mean, m2;
        row_stats(v, Dh, 32, &mean, &m2);
        float rstd = stats_rstd(m2, Dh, eps);
        for (int64_t d = 0; d < Dh; ++d) {
            float u = rstd * (v[d] - mean);
            out[(r - row_begin) * Dh + d] =
                store16(fmaf(load16(w[d], dtype), u, load16(bias[d], dtype)), dtype);
        }
    }
    return 0;
}

/* One tensor: rows of Dh contiguous values, RMSNorm with a weight on 32
 * logical lanes: rstd = rsqrt_cr(ss / Dh + eps) with ss from row_sumsq,
 * u = rstd * x, out = round16(w * u) (binary32 products, one storage
 * rounding).  Rows [row_begin, row_end); row r goes to
 * out + (r - row_begin) * Dh.  Returns -1 unless 0 < Dh <= 128 and
 * Dh % 4 == 0. */
int oracle_qk_rmsnorm(uint16_t *out, const uint16_t *in, int64_t rows, int64_t Dh,
                      const uint16_t *w, float eps, int dtype, int64_t row_begin, int64_t row_end) {
    if (Dh <= 0 || Dh > 128 || Dh % 4) return -1;
    float v[128];
    for (int64_t r = row_begin; r < row_end && r < rows; ++r) {
        const uint16_t *xr = in + r * Dh;
        for (int64_t d = 0; d < Dh; ++d) v[d] = load16(xr[d], dtype);
        float rstd = rms_rstd(row_sumsq(v, Dh, 32), Dh, eps);
        for (int64_t d = 0; d < Dh; ++d) {
            float u = rstd * v[d];
            out[(r - row_begin) * Dh + d] = store16(load16(w[d], dtype) * u, dtype);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* residual_gate_add                                                    */
/* ------------------------------------------------------------------ */

/* out[b, n, d] = round16(x + round16(gate[b, d] * y)), x, y contiguous
 * (B, N, D); gate row b at gate + b * s_gate_b.  Rows r = b*N + n in
 * [row_begin, row_end); row r goes to out + (r - row_begin) * D. */
int oracle_residual_gate_add(uint16_t *out, const uint16_t *x, const uint16_t *gate,
                             int64_t s_gate_b, const uint16_t *y, int64_t B, int64_t N,
                             int64_t D, int dtype, int64_t row_begin, int64_t row_end) {
    for (int64_t r = row_begin; r < row_end && r < B * N; ++r) {
        const uint16_t *g = gate + (r / N) * s_gate_b;
        for (int64_t d = 0; d < D; ++d)
            out[(r - row_begin) * D + d] = store16(gate_add(load16(x[r * D + d], dtype), g[d], y[r * D + d], dtype), dtype);
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* bias + tanh-GELU                                                     */
/* ------------------------------------------------------------------ */

/* G(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))), evaluated as
 * v / (1 + exp(-2 z)) with z = sqrt(2/pi) (v + 0.044715 v^3) (the same real
 * number, without the cancellation of 1 + tanh for z << 0), in long double,
 * then rounded once to binary32.  The rounding is certified: if the long
 * double value lies within 2^-50 (relative) of a binary32 rounding boundary
 * the oracle refuses (abort) instead of guessing. */
static float gelu_f32(float vf) {
    if (isnan(vf)) return NAN;
    if (isinf(vf)) return vf > 0 ? INFINITY : NAN; /* -inf * 0 in the eager formula */
    long double v = vf;
    const long double k0 = 0.797884560802865355879892119868763737L; /* sqrt(2/pi) */
    const long double k1 = 0.044715L;
    long double z = k0 * (v + k1 * v * v * v);
    long double g = v / (1.0L + expl(-2.0L * z));
    float f = (float)g;
    if (g != 0.0L && isfinite(f)) {
        float up = nextafterf(f, INFINITY), dn = nextafterf(f, -INFINITY);
        long double mu = ((long double)f + (long double)up) / 2.0L;
        long double md = ((long double)f + (long double)dn) / 2.0L;
        long double tol = fabsl(g) * 0x1.0p-50L;
        if (fabsl(g - mu) < tol || fabsl(g - md) < tol) {
            fprintf(stderr, "oracle gelu: uncertified rounding at v=%a\n", (double)vf);
            abort();
        }
    }
    return f;
}

/* table[h] = round16(G(value of pattern h)) for all 65536 patterns */
int oracle_gelu_table(uint16_t *table, int dtype) {
    for (uint32_t h = 0; h < 65536u; ++h) {
        float v = load16((uint16_t)h, dtype);
        table[h] = store16(gelu_f32(v), dtype);
    }
    return 0;
}

static uint16_t *g_tables[2];

/* out[r, c] = round16(G(round16(x[r, c] + bias[c]))) for rows
 * [row_begin, row_end); x contiguous (rows, width); row r goes to
 * out + (r - row_begin) * width. */
int oracle_bias_gelu_tanh(uint16_t *out, const uint16_t *x, const uint16_t *bias, int64_t rows,
                          int64_t width, int dtype, int64_t row_begin, int64_t row_end) {
    dtype = dtype ? 1 : 0;
    if (!g_tables[dtype]) {
        uint16_t *t = (uint16_t *)malloc(65536 * sizeof(uint16_t));
        if (!t) return -2;
        oracle_gelu_table(t, dtype);
        g_tables[dtype] = t;
    }
    const uint16_t *tab = g_tables[dtype];
    for (int64_t r = row_begin; r < row_end && r < rows; ++r)
        for (int64_t c = 0; c < width; ++c) {
            uint16_t v = store16(load16(x[r * width + c], dtype) + load16(bias[c], dtype), dtype);
            out[(r - row_begin) * width + c] = tab[v];
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* temb_table_slices                                                    */
/* ------------------------------------------------------------------ */

/* Element of a 16-bit or binary32 array as binary32 (exact): dtype 0 bf16,
 * 1 fp16, 2 binary32. */
static float load_any(const void *p, int64_t i, int dtype) {
    if (dtype == 2) return ((const float *)p)[i];
    return load16(((const uint16_t *)p)[i], dtype);
}

/* out_k[b, s, d] = table[k, d] + temb[b, s, k, d] in binary32 (one IEEE
 * addition of the exact binary32 values of both operands), for the K
 * chunks of a (B, S, K, D) temb, each written to its own contiguous
 * (B, S, D) slice at out + k * s_out_k.  table (K, D) and temb contiguous.
 * Returns -1 for a bad dtype or size. */
int oracle_temb_table_slices(float *out, int64_t s_out_k, const void *table, int table_dtype,
                             const void *temb, int temb_dtype, int64_t B, int64_t S, int64_t K,
                             int64_t D) {
    if (table_dtype < 0 || table_dtype > 2 || temb_dtype < 0 || temb_dtype > 2) return -1;
    if (B < 1 || S < 1 || K < 1 || D < 1) return -1;
    for (int64_t k = 0; k < K; ++k)
        for (int64_t bs = 0; bs < B * S; ++bs)
            for (int64_t d = 0; d < D; ++d)
                out[k * s_out_k + bs * D + d] =
                    load_any(table, k * D + d, table_dtype) + load_any(temb, (bs * K + k) * D + d, temb_dtype);
    return 0;
}

/* ------------------------------------------------------------------ */
/* static FP8 (e4m3, finite-only) quantisation                          */
/* ------------------------------------------------------------------ */

/* binary32 -> fp8 e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; no infinities; 0x7F / 0xFF are NaN; largest finite 448), round to
 * nearest even with saturation: |f| beyond 448, infinities included, give
 * +-448; NaN gives 0x7F.  Written from the format definition: the result is
 * the nearest multiple of the quantum of f's binade (2^(e-3) for
 * 2^e <= |f| < 2^(e+1), e >= -6; 2^-9 below 2^-6), ties to the even
 * multiple. */
static uint8_t f32_to_e4m3_sat(float f) {
    if (isnan(f)) return 0x7f;
    uint8_t sign = signbit(f) ? 0x80 : 0x00;
    double a = fabs((double)f);
    if (a >= 448.0) return sign | 0x7e;
    int e;
    frexp(a, &e);                 /* a = m * 2^e, m in [0.5, 1) (a > 0) */
    int ex = (a == 0.0) ? -6 : e - 1;
    if (ex < -6) ex = -6;         /* subnormal quantum 2^-9 */
    double quantum = ldexp(1.0, ex - 3);
    double q = a / quantum;       /* exact: a has 24 significant bits */
    double r = floor(q), frac = q - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    double v = r * quantum;       /* <= 448: values from 448 up returned above */
    if (v == 0.0) return sign;
    int ve;
    frexp(v, &ve);
    int E = ve - 1;               /* binade of the rounded value */
    if (E < -6) return sign | (uint8_t)(v / ldexp(1.0, -9));            /* subnormal code */
    int mant = (int)(v / ldexp(1.0, E - 3)) - 8;                        /* 0..7 */
    return sign | (uint8_t)(((E + 7) << 3) | mant);
}

/* out8[i] = e4m3(value(y[i]) / qscale), y storage values (dtype 0 bf16,
 * 1 fp16), one IEEE binary32 division, then f32_to_e4m3_sat. */
int oracle_quant_e4m3(uint8_t *out8, const uint16_t *y, int64_t n, float qscale, int dtype) {
    for (int64_t i = 0; i < n; ++i) out8[i] = f32_to_e4m3_sat(load16(y[i], dtype) / qscale);
    return 0;
}

/* every binary32 input of a pin through the encoder */
void oracle_f32_to_e4m3_array(const float *in, uint8_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3_sat(in[i]);
}

/* ------------------------------------------------------------------ */
/* small exports for the oracle's own pins                              */
/* ------------------------------------------------------------------ */

void oracle_f32_to_16(const float *in, uint16_t *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = store16(in[i], dtype);
}
void oracle_16_to_f32(const uint16_t *in, float *out, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) out[i] = load16(in[i], dtype);
}
void oracle_rsqrt_cr_array(const float *in, float *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_rsqrt_cr(in[i]);
}
/* RMSNorm sum of squares on L lanes (128 or 32) of one binary32 row */
int oracle_row_sumsq(const float *x, int64_t D, int L, float *ss) {
    if (D <= 0 || D % 4 || (L != 128 && L != 32) || (L == 32 && D > 128)) return -1;
    *ss = row_sumsq(x, D, L);
    return 0;
}
/* row statistics on L lanes (128 or 32) of one binary32 row */
int oracle_row_stats(const float *x, int64_t D, int L, float *mean, float *m2) {
    if (D <= 0 || D % 4 || (L != 128 && L != 32) || (L == 32 && D > 128)) return -1;
    row_stats(x, D, L, mean, m2);
    return 0;
}
