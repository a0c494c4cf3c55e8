// C ABI of the library: argument validation, per-device state, dispatch.
// Declared in include/adaln.h; every entry point is extern "C", takes plain
// pointers and sizes, and validates everything on the host before the first
// CUDA call.
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <initializer_list>
#include <mutex>

#include "../../include/adaln.h"
#include "kernels.h"

using namespace adaln;

namespace {

constexpr int kMaxDevices = kApiMaxDevices;

struct DevState {
    DeviceInfo info;
    bool have_info = false;
    void *gelu = nullptr;  // 2 x 65536 storage values: bf16 table then fp16 table
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
thread_local char g_err[256] = "";

adaln_status cuda_fail(cudaError_t e) {
    snprintf(g_err, sizeof(g_err), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return ADALN_E_CUDA;
}

adaln_status current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (*dev < 0 || *dev >= kMaxDevices) {
        snprintf(g_err, sizeof(g_err), "device ordinal %d beyond %d", *dev, kMaxDevices);
        return ADALN_E_CUDA;
    }
    return ADALN_OK;
}

// device properties, cached (the caller holds no lock)
adaln_status device_info(int dev, DeviceInfo *out) {
    std::lock_guard<std::mutex> lk(g_mu);
    DevState &d = g_dev[dev];
    if (!d.have_info) {
        int sms = 0, smem = 0, l2 = 0;
        cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        if (e != cudaSuccess) return cuda_fail(e);
        d.info.device = dev;
        d.info.sms = sms;
        d.info.max_smem_optin = smem;
        d.info.l2_bytes = l2;
        d.have_info = true;
    }
    *out = d.info;
    return ADALN_OK;
}

// builds the GELU tables of the current device (g_mu held by the caller)
adaln_status build_tables_locked(int dev) {
    DevState &d = g_dev[dev];
    if (d.gelu) return ADALN_OK;
    void *buf = nullptr;
    cudaError_t e = cudaMalloc(&buf, 2 * 65536 * sizeof(uint16_t));
    if (e != cudaSuccess) return cuda_fail(e);
    cudaStream_t s = nullptr;
    e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = launch_gelu_table_init(buf, 0, s);
    if (e == cudaSuccess) e = launch_gelu_table_init((uint16_t *)buf + 65536, 1, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (s) cudaStreamDestroy(s);
    if (e != cudaSuccess) {
        cudaFree(buf);
        return cuda_fail(e);
    }
    d.gelu = buf;
    return ADALN_OK;
}

bool finite_nonneg(float v) { return isfinite(v) && v >= 0.0f; }

// strides beyond 2^46 elements describe no real buffer and would overflow the
// byte extents the overlap checks compute
constexpr int64_t kMaxStride = (int64_t)1 << 46;
bool strides_ok(std::initializer_list<int64_t> ss) {
    for (int64_t v : ss)
        if (v < 0 || v > kMaxStride) return false;
    return true;
}
bool al2(const void *p) { return ((uintptr_t)p & 1u) == 0; }
bool al8(const void *p) { return ((uintptr_t)p & 7u) == 0; }

// [a, a+na) and [b, b+nb) in bytes intersect
bool overlap(const void *a, int64_t na, const void *b, int64_t nb) {
    const uintptr_t pa = (uintptr_t)a, pb = (uintptr_t)b;
    return pa < pb + (uintptr_t)nb && pb < pa + (uintptr_t)na;
}

// ------------------------------------------------------------ checks

adaln_status check_ln(const void *out, const void *x, int64_t B, int64_t N, int64_t D, int64_t sxB,
                      int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b, const void *shift,
                      int64_t s_shift_b, float eps, int dtype, uint32_t flags) {
    if (dtype != ADALN_BF16 && dtype != ADALN_FP16) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (!out || !x || !scale || !shift) return ADALN_E_NULL;
    if (B < 1 || N < 1 || D < 4 || D > 65536 || D % 4 != 0) return ADALN_E_SHAPE;
    if (B > ((int64_t)1 << 40) / N || B * N > ((int64_t)1 << 46) / D) return ADALN_E_SHAPE;
    if (!strides_ok({sxB, sxN, sxD, s_scale_b, s_shift_b})) return ADALN_E_STRIDE;
    if (!finite_nonneg(eps)) return ADALN_E_VALUE;
    if (!al2(out) || !al2(x) || !al2(scale) || !al2(shift)) return ADALN_E_ALIGN;
    const int64_t out_bytes = 2 * B * N * D;
    const int64_t x_bytes = 2 * ((B - 1) * sxB + (N - 1) * sxN + (D - 1) * sxD + 1);
    const bool x_contig = sxD == 1 && (N == 1 || sxN == D) && (B == 1 || sxB == N * D);
    if (overlap(out, out_bytes, x, x_bytes) && !(out == x && x_contig)) return ADALN_E_OVERLAP;
    if (overlap(out, out_bytes, scale, 2 * ((B - 1) * s_scale_b + D))) return ADALN_E_OVERLAP;
    if (overlap(out, out_bytes, shift, 2 * ((B - 1) * s_shift_b + D))) return ADALN_E_OVERLAP;
    return ADALN_OK;
}

adaln_status check_qk(const void *q_out, const void *q, int64_t rows_q, const void *k_out, const void *k,
                      int64_t rows_k, int64_t Dh, const void *wq, const void *bq, const void *wk,
                      const void *bk, float eps, int dtype, uint32_t flags) {
    if (dtype != ADALN_BF16 && dtype != ADALN_FP16) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (rows_q < 0 || rows_k < 0 || rows_q + rows_k < 1) return ADALN_E_SHAPE;
    if (Dh < 4 || Dh > 128 || Dh % 4 != 0) return ADALN_E_SHAPE;
    if (rows_q > ((int64_t)1 << 46) / Dh || rows_k > ((int64_t)1 << 46) / Dh) return ADALN_E_SHAPE;
    if (rows_q > 0 && (!q_out || !q || !wq || !bq)) return ADALN_E_NULL;
    if (rows_k > 0 && (!k_out || !k || !wk || !bk)) return ADALN_E_NULL;
    if (!finite_nonneg(eps)) return ADALN_E_VALUE;
    const void *ptrs[] = {rows_q ? q_out : nullptr, rows_q ? q : nullptr, rows_q ? wq : nullptr,
                          rows_q ? bq : nullptr, rows_k ? k_out : nullptr, rows_k ? k : nullptr,
                          rows_k ? wk : nullptr, rows_k ? bk : nullptr};
    for (const void *p : ptrs)
        if (p && !al8(p)) return ADALN_E_ALIGN;
    const int64_t qb = 2 * rows_q * Dh, kb = 2 * rows_k * Dh, vb = 2 * Dh;
    if (rows_q) {
        if (overlap(q_out, qb, q, qb) && q_out != q) return ADALN_E_OVERLAP;
        if (overlap(q_out, qb, wq, vb) || overlap(q_out, qb, bq, vb)) return ADALN_E_OVERLAP;
        if (rows_k && (overlap(q_out, qb, k, kb) || overlap(q_out, qb, k_out, kb) ||
                       overlap(q_out, qb, wk, vb) || overlap(q_out, qb, bk, vb)))
            return ADALN_E_OVERLAP;
    }
    if (rows_k) {
        if (overlap(k_out, kb, k, kb) && k_out != k) return ADALN_E_OVERLAP;
        if (overlap(k_out, kb, wk, vb) || overlap(k_out, kb, bk, vb)) return ADALN_E_OVERLAP;
        if (rows_q && (overlap(k_out, kb, q, qb) || overlap(k_out, kb, wq, vb) || overlap(k_out, kb, bq, vb)))
            return ADALN_E_OVERLAP;
    }
    return ADALN_OK;
}

adaln_status check_gate(const void *out, const void *x, const void *gate, int64_t s_gate_b, const void *y,
                        int64_t B, int64_t N, int64_t D, int dtype, uint32_t flags) {
    if (dtype != ADALN_BF16 && dtype != ADALN_FP16) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (!out || !x || !gate || !y) return ADALN_E_NULL;
    if (B < 1 || N < 1 || D < 1) return ADALN_E_SHAPE;
    if (B > ((int64_t)1 << 40) / N || B * N > ((int64_t)1 << 46) / D) return ADALN_E_SHAPE;
    if (!strides_ok({s_gate_b})) return ADALN_E_STRIDE;
    if (!al2(out) || !al2(x) || !al2(gate) || !al2(y)) return ADALN_E_ALIGN;
    const int64_t nb = 2 * B * N * D;
    if (overlap(out, nb, x, nb) && out != x) return ADALN_E_OVERLAP;
    if (overlap(out, nb, y, nb) && out != y) return ADALN_E_OVERLAP;
    if (overlap(out, nb, gate, 2 * ((B - 1) * s_gate_b + D))) return ADALN_E_OVERLAP;
    return ADALN_OK;
}

// r_out = x + gate * y and out = LN(r_out) * (1 + scale) + shift, all (B, N, D) contiguous
adaln_status check_residual_ln(const void *r_out, const void *out, const void *x, const void *gate, int64_t s_gate_b,
                               const void *y, int64_t B, int64_t N, int64_t D, const void *scale,
                               int64_t s_scale_b, const void *shift, int64_t s_shift_b, float eps, int dtype,
                               uint32_t flags) {
    adaln_status st = check_gate(r_out, x, gate, s_gate_b, y, B, N, D, dtype, flags);
    if (st != ADALN_OK) return st;
    st = check_ln(out, r_out, B, N, D, N * D, D, 1, scale, s_scale_b, shift, s_shift_b, eps, dtype, flags);
    if (st != ADALN_OK) return st;
    const int64_t nb = 2 * B * N * D;
    if (overlap(out, nb, r_out, nb) || overlap(out, nb, x, nb) || overlap(out, nb, y, nb) ||
        overlap(out, nb, gate, 2 * ((B - 1) * s_gate_b + D)))
        return ADALN_E_OVERLAP;
    if (overlap(r_out, nb, scale, 2 * ((B - 1) * s_scale_b + D)) ||
        overlap(r_out, nb, shift, 2 * ((B - 1) * s_shift_b + D)))
        return ADALN_E_OVERLAP;
    return ADALN_OK;
}

// bytes from p to one past the last element of a (B, N, D) operand with
// strides (sb, sn, sd)
int64_t extent(int64_t B, int64_t N, int64_t D, int64_t sb, int64_t sn, int64_t sd) {
    return 2 * ((B - 1) * sb + (N - 1) * sn + (D - 1) * sd + 1);
}

// the general norm + modulate: norm 0 LayerNorm / 1 RMSNorm, optional
// residual gate (gate != NULL), per-sample or per-token operand rows
adaln_status check_norm(int norm, const void *r_out, const void *out, const void *x, int64_t B, int64_t N,
                        int64_t D, int64_t sxB, int64_t sxN, int64_t sxD, const void *gate, int64_t s_gate_b,
                        int64_t s_gate_n, int64_t s_gate_d, const void *y, const void *scale, int64_t s_scale_b,
                        int64_t s_scale_n, const void *shift, int64_t s_shift_b, int64_t s_shift_n, float eps,
                        int dtype, uint32_t flags) {
    if (dtype != ADALN_BF16 && dtype != ADALN_FP16) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (norm != ADALN_NORM_LAYER && norm != ADALN_NORM_RMS) return ADALN_E_VALUE;
    if (!out || !x || !scale || !shift) return ADALN_E_NULL;
    if (gate && (!y || !r_out)) return ADALN_E_NULL;
    if (B < 1 || N < 1 || D < 4 || D > 65536 || D % 4 != 0) return ADALN_E_SHAPE;
    if (B > ((int64_t)1 << 40) / N || B * N > ((int64_t)1 << 46) / D) return ADALN_E_SHAPE;
    if (!strides_ok({sxB, sxN, sxD, s_scale_b, s_scale_n, s_shift_b, s_shift_n})) return ADALN_E_STRIDE;
    if (!finite_nonneg(eps)) return ADALN_E_VALUE;
    if (!al2(out) || !al2(x) || !al2(scale) || !al2(shift)) return ADALN_E_ALIGN;
    const int64_t nb = 2 * B * N * D;
    const bool x_contig = sxD == 1 && (N == 1 || sxN == D) && (B == 1 || sxB == N * D);
    const int64_t x_bytes = extent(B, N, D, sxB, sxN, sxD);
    const int64_t sc_bytes = extent(B, N, D, s_scale_b, s_scale_n, 1);
    const int64_t sh_bytes = extent(B, N, D, s_shift_b, s_shift_n, 1);
    if (overlap(out, nb, scale, sc_bytes) || overlap(out, nb, shift, sh_bytes)) return ADALN_E_OVERLAP;
    if (!gate) {
        if (overlap(out, nb, x, x_bytes) && !(out == x && x_contig)) return ADALN_E_OVERLAP;
        return ADALN_OK;
    }
    if (!strides_ok({s_gate_b, s_gate_n}) || (s_gate_d != 0 && s_gate_d != 1)) return ADALN_E_STRIDE;
    if (!x_contig) return ADALN_E_STRIDE;
    if (!al2(gate) || !al2(y) || !al2(r_out)) return ADALN_E_ALIGN;
    const int64_t g_bytes = extent(B, N, D, s_gate_b, s_gate_n, s_gate_d);
    if (overlap(out, nb, x, nb) || overlap(out, nb, y, nb) || overlap(out, nb, r_out, nb) ||
        overlap(out, nb, gate, g_bytes))
        return ADALN_E_OVERLAP;
    if (overlap(r_out, nb, x, nb) && r_out != x) return ADALN_E_OVERLAP;
    if (overlap(r_out, nb, y, nb) && r_out != y) return ADALN_E_OVERLAP;
    if (overlap(r_out, nb, gate, g_bytes) || overlap(r_out, nb, scale, sc_bytes) ||
        overlap(r_out, nb, shift, sh_bytes))
        return ADALN_E_OVERLAP;
    return ADALN_OK;
}

LnArgs norm_args(int norm, void *r_out, void *out, const void *x, int64_t B, int64_t N, int64_t D, int64_t sxB,
                 int64_t sxN, int64_t sxD, const void *gate, int64_t s_gate_b, int64_t s_gate_n, int64_t s_gate_d,
                 const void *y, const void *scale, int64_t s_scale_b, int64_t s_scale_n, const void *shift,
                 int64_t s_shift_b, int64_t s_shift_n, float eps) {
    LnArgs a{out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps};
    a.s_scale_n = s_scale_n;
    a.s_shift_n = s_shift_n;
    a.norm = norm;
    if (gate) {
        a.gate = gate;
        a.s_gate_b = s_gate_b;
        a.s_gate_n = s_gate_n;
        a.s_gate_d = s_gate_d;
        a.y = y;
        a.r_out = r_out;
    }
    return a;
}

// LayerNorm + modulate into static FP8: check_ln's rules with 1-byte outputs
adaln_status check_ln_fp8(const void *out, const void *qscale, const void *x, int64_t B, int64_t N, int64_t D,
                          int64_t sxB, int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b,
                          const void *shift, int64_t s_shift_b, float eps, int dtype, uint32_t flags) {
    if (dtype != ADALN_BF16 && dtype != ADALN_FP16) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (!out || !qscale || !x || !scale || !shift) return ADALN_E_NULL;
    if (B < 1 || N < 1 || D < 4 || D > 65536 || D % 4 != 0) return ADALN_E_SHAPE;
    if (B > ((int64_t)1 << 40) / N || B * N > ((int64_t)1 << 46) / D) return ADALN_E_SHAPE;
    if (!strides_ok({sxB, sxN, sxD, s_scale_b, s_shift_b})) return ADALN_E_STRIDE;
    if (!finite_nonneg(eps)) return ADALN_E_VALUE;
    if (!al2(x) || !al2(scale) || !al2(shift) || ((uintptr_t)qscale & 3u)) return ADALN_E_ALIGN;
    const int64_t nb = B * N * D;
    if (overlap(out, nb, x, extent(B, N, D, sxB, sxN, sxD)) ||
        overlap(out, nb, scale, extent(B, 1, D, s_scale_b, 0, 1)) ||
        overlap(out, nb, shift, extent(B, 1, D, s_shift_b, 0, 1)) || overlap(out, nb, qscale, 4))
        return ADALN_E_OVERLAP;
    return ADALN_OK;
}

adaln_status check_temb(const void *out, int64_t s_out_k, const void *table, int table_dtype, const void *temb,
                        int temb_dtype, int64_t B, int64_t S, int64_t K, int64_t D, uint32_t flags) {
    auto ok_dt = [](int d) { return d == ADALN_BF16 || d == ADALN_FP16 || d == ADALN_FP32; };
    if (!ok_dt(table_dtype) || !ok_dt(temb_dtype)) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (!out || !table || !temb) return ADALN_E_NULL;
    if (B < 1 || S < 1 || K < 1 || D < 1 || K > 65536 || D > 65536) return ADALN_E_SHAPE;
    if (B > ((int64_t)1 << 40) / S || B * S > ((int64_t)1 << 44) / (K * D)) return ADALN_E_SHAPE;
    const int64_t slice = B * S * D;
    if (K > 1 && (s_out_k < slice || s_out_k > ((int64_t)1 << 46) / K)) return ADALN_E_STRIDE;
    const int te = table_dtype == ADALN_FP32 ? 4 : 2, ee = temb_dtype == ADALN_FP32 ? 4 : 2;
    if (((uintptr_t)out & 3u) || ((uintptr_t)table % te) || ((uintptr_t)temb % ee)) return ADALN_E_ALIGN;
    const int64_t out_bytes = 4 * ((K - 1) * (K > 1 ? s_out_k : 0) + slice);
    if (overlap(out, out_bytes, table, (int64_t)te * K * D) || overlap(out, out_bytes, temb, ee * slice * K))
        return ADALN_E_OVERLAP;
    return ADALN_OK;
}

adaln_status check_gelu(const void *out, const void *x, const void *bias, int64_t rows, int64_t width,
                        int dtype, uint32_t flags) {
    if (dtype != ADALN_BF16 && dtype != ADALN_FP16) return ADALN_E_DTYPE;
    if (flags & ~ADALN_FLAG_PDL) return ADALN_E_VALUE;
    if (!out || !x || !bias) return ADALN_E_NULL;
    if (rows < 1 || width < 1 || rows > ((int64_t)1 << 46) / width) return ADALN_E_SHAPE;
    if (!al2(out) || !al2(x) || !al2(bias)) return ADALN_E_ALIGN;
    const int64_t nb = 2 * rows * width;
    if (overlap(out, nb, x, nb) && out != x) return ADALN_E_OVERLAP;
    if (overlap(out, nb, bias, 2 * width)) return ADALN_E_OVERLAP;
    return ADALN_OK;
}

adaln_status finish_launch(cudaError_t e) { return e == cudaSuccess ? ADALN_OK : cuda_fail(e); }

}  // namespace

namespace adaln {

adaln_status api_current_device(int *dev) { return current_device(dev); }
adaln_status api_device_info(int dev, DeviceInfo *out) { return device_info(dev, out); }
adaln_status api_cuda_fail(cudaError_t e) { return cuda_fail(e); }
adaln_status api_fail_msg(const char *msg) {
    snprintf(g_err, sizeof(g_err), "%s", msg);
    return ADALN_E_CUDA;
}

int blocks_per_sm_cached(const void *kernel, int threads, size_t smem) {
    struct Entry {
        const void *k;
        int threads;
        size_t smem;
        int n;
    };
    static Entry cache[128];
    static int used = 0;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].k == kernel && cache[i].threads == threads && cache[i].smem == smem) return cache[i].n;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1)
        n = 1;
    if (used < 128) cache[used++] = Entry{kernel, threads, smem, n};
    return n;
}

}  // namespace adaln

extern "C" {

const char *adaln_status_str(int status) {
    switch (status) {
        case ADALN_OK: return "ADALN_OK";
        case ADALN_E_NULL: return "ADALN_E_NULL: a required pointer is NULL";
        case ADALN_E_DTYPE: return "ADALN_E_DTYPE: dtype must be ADALN_BF16 or ADALN_FP16 (or ADALN_FP32 where allowed)";
        case ADALN_E_SHAPE: return "ADALN_E_SHAPE: a size is out of range";
        case ADALN_E_ALIGN: return "ADALN_E_ALIGN: a pointer is not aligned";
        case ADALN_E_STRIDE: return "ADALN_E_STRIDE: a stride is negative";
        case ADALN_E_VALUE: return "ADALN_E_VALUE: eps negative or not finite, or unknown flags";
        case ADALN_E_OVERLAP: return "ADALN_E_OVERLAP: an output overlaps an input";
        case ADALN_E_CUDA: return "ADALN_E_CUDA: a CUDA call failed";
    }
    return "unknown adaln_status";
}

const char *adaln_last_cuda_error(void) { return g_err; }

int adaln_version(void) { return 10000; }

adaln_status adaln_init(int device) {
    if (device < 0 || device >= kMaxDevices) return ADALN_E_VALUE;
    int prev = 0;
    cudaError_t e = cudaGetDevice(&prev);
    if (e != cudaSuccess) return cuda_fail(e);
    if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return cuda_fail(e);
    DeviceInfo info;
    adaln_status st = device_info(device, &info);
    if (st == ADALN_OK) {
        std::lock_guard<std::mutex> lk(g_mu);
        st = build_tables_locked(device);
    }
    if (prev != device) cudaSetDevice(prev);
    return st;
}

adaln_status adaln_shutdown(void) {
    std::lock_guard<std::mutex> lk(g_mu);
    int prev = 0;
    cudaGetDevice(&prev);
    adaln_status st = ADALN_OK;
    for (int d = 0; d < kMaxDevices; ++d) {
        if (!g_dev[d].gelu) continue;
        cudaSetDevice(d);
        cudaError_t e = cudaFree(g_dev[d].gelu);
        if (e != cudaSuccess) st = cuda_fail(e);
        g_dev[d].gelu = nullptr;
    }
    cudaSetDevice(prev);
    return st;
}

adaln_status adaln_can_ln_modulate(const void *out, const void *x, int64_t B, int64_t N, int64_t D,
                                   int64_t sxB, int64_t sxN, int64_t sxD, const void *scale,
                                   int64_t s_scale_b, const void *shift, int64_t s_shift_b, float eps,
                                   int dtype, uint32_t flags) {
    return check_ln(out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps, dtype, flags);
}

int adaln_ln_modulate_variant(const void *out, const void *x, int64_t B, int64_t N, int64_t D, int64_t sxB,
                              int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b,
                              const void *shift, int64_t s_shift_b, float eps, int dtype, uint32_t flags) {
    adaln_status st =
        check_ln(out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps, dtype, flags);
    if (st != ADALN_OK) return -(int)st;
    LnArgs a{(void *)out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps};
    const int path = ln_modulate_path(a);
    if (path == LN_PATH_TOKENS) {
        // the TMA tile kernel needs a device (its shared memory) and the driver
        int dev;
        DeviceInfo info;
        if (current_device(&dev) == ADALN_OK && device_info(dev, &info) == ADALN_OK &&
            ln_tokens_tma_ready(a, info))
            return LN_PATH_TOKENS_TMA;
    }
    return path;
}

adaln_status adaln_ln_modulate(void *out, const void *x, int64_t B, int64_t N, int64_t D, int64_t sxB,
                               int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b,
                               const void *shift, int64_t s_shift_b, float eps, int dtype, uint32_t flags,
                               void *stream) {
    adaln_status st =
        check_ln(out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    LnArgs a{out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps};
    return finish_launch(
        launch_ln_modulate(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_residual_gate_ln_modulate(const void *r_out, const void *out, const void *x,
                                                 const void *gate, int64_t s_gate_b, const void *y, int64_t B,
                                                 int64_t N, int64_t D, const void *scale, int64_t s_scale_b,
                                                 const void *shift, int64_t s_shift_b, float eps, int dtype,
                                                 uint32_t flags) {
    return check_residual_ln(r_out, out, x, gate, s_gate_b, y, B, N, D, scale, s_scale_b, shift, s_shift_b, eps,
                             dtype, flags);
}

adaln_status adaln_residual_gate_ln_modulate(void *r_out, void *out, const void *x, const void *gate,
                                             int64_t s_gate_b, const void *y, int64_t B, int64_t N, int64_t D,
                                             const void *scale, int64_t s_scale_b, const void *shift,
                                             int64_t s_shift_b, float eps, int dtype, uint32_t flags, void *stream) {
    adaln_status st = check_residual_ln(r_out, out, x, gate, s_gate_b, y, B, N, D, scale, s_scale_b, shift,
                                        s_shift_b, eps, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    LnArgs a{out, x, B, N, D, N * D, D, 1, scale, s_scale_b, shift, s_shift_b, eps};
    a.gate = gate;
    a.s_gate_b = s_gate_b;
    a.y = y;
    a.r_out = r_out;
    return finish_launch(launch_norm_scale_shift(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_norm_scale_shift(int norm, const void *r_out, const void *out, const void *x, int64_t B,
                                        int64_t N, int64_t D, int64_t sxB, int64_t sxN, int64_t sxD,
                                        const void *gate, int64_t s_gate_b, int64_t s_gate_n, int64_t s_gate_d,
                                        const void *y, const void *scale, int64_t s_scale_b, int64_t s_scale_n,
                                        const void *shift, int64_t s_shift_b, int64_t s_shift_n, float eps,
                                        int dtype, uint32_t flags) {
    return check_norm(norm, r_out, out, x, B, N, D, sxB, sxN, sxD, gate, s_gate_b, s_gate_n, s_gate_d, y, scale,
                      s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps, dtype, flags);
}

int adaln_norm_scale_shift_variant(int norm, const void *r_out, const void *out, const void *x, int64_t B, int64_t N,
                                   int64_t D, int64_t sxB, int64_t sxN, int64_t sxD, const void *gate,
                                   int64_t s_gate_b, int64_t s_gate_n, int64_t s_gate_d, const void *y,
                                   const void *scale, int64_t s_scale_b, int64_t s_scale_n, const void *shift,
                                   int64_t s_shift_b, int64_t s_shift_n, float eps, int dtype, uint32_t flags) {
    adaln_status st = check_norm(norm, r_out, out, x, B, N, D, sxB, sxN, sxD, gate, s_gate_b, s_gate_n, s_gate_d, y,
                                 scale, s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps, dtype, flags);
    if (st != ADALN_OK) return -(int)st;
    const LnArgs a = norm_args(norm, (void *)r_out, (void *)out, x, B, N, D, sxB, sxN, sxD, gate, s_gate_b, s_gate_n,
                               s_gate_d, y, scale, s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps);
    const int path = ln_modulate_path(a);
    if (path == LN_PATH_TOKENS) {
        int dev;
        DeviceInfo info;
        if (current_device(&dev) == ADALN_OK && device_info(dev, &info) == ADALN_OK && ln_tokens_tma_ready(a, info))
            return LN_PATH_TOKENS_TMA;
    }
    return path;
}

adaln_status adaln_norm_scale_shift(int norm, void *r_out, void *out, const void *x, int64_t B, int64_t N, int64_t D,
                                    int64_t sxB, int64_t sxN, int64_t sxD, const void *gate, int64_t s_gate_b,
                                    int64_t s_gate_n, int64_t s_gate_d, const void *y, const void *scale,
                                    int64_t s_scale_b, int64_t s_scale_n, const void *shift, int64_t s_shift_b,
                                    int64_t s_shift_n, float eps, int dtype, uint32_t flags, void *stream) {
    adaln_status st = check_norm(norm, r_out, out, x, B, N, D, sxB, sxN, sxD, gate, s_gate_b, s_gate_n, s_gate_d, y,
                                 scale, s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    const LnArgs a = norm_args(norm, r_out, out, x, B, N, D, sxB, sxN, sxD, gate, s_gate_b, s_gate_n, s_gate_d, y,
                               scale, s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps);
    return finish_launch(launch_norm_scale_shift(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_rmsnorm_scale_shift(const void *out, const void *x, int64_t B, int64_t N, int64_t D,
                                           int64_t sxB, int64_t sxN, int64_t sxD, const void *scale,
                                           int64_t s_scale_b, int64_t s_scale_n, const void *shift,
                                           int64_t s_shift_b, int64_t s_shift_n, float eps, int dtype,
                                           uint32_t flags) {
    return check_norm(ADALN_NORM_RMS, nullptr, out, x, B, N, D, sxB, sxN, sxD, nullptr, 0, 0, 1, nullptr, scale,
                      s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps, dtype, flags);
}

adaln_status adaln_rmsnorm_scale_shift(void *out, const void *x, int64_t B, int64_t N, int64_t D, int64_t sxB,
                                       int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b,
                                       int64_t s_scale_n, const void *shift, int64_t s_shift_b, int64_t s_shift_n,
                                       float eps, int dtype, uint32_t flags, void *stream) {
    return adaln_norm_scale_shift(ADALN_NORM_RMS, nullptr, out, x, B, N, D, sxB, sxN, sxD, nullptr, 0, 0, 1, nullptr,
                                  scale, s_scale_b, s_scale_n, shift, s_shift_b, s_shift_n, eps, dtype, flags,
                                  stream);
}

adaln_status adaln_can_qk_head_layernorm(const void *q_out, const void *q, int64_t rows_q, const void *k_out,
                                         const void *k, int64_t rows_k, int64_t Dh, const void *wq,
                                         const void *bq, const void *wk, const void *bk, float eps, int dtype,
                                         uint32_t flags) {
    return check_qk(q_out, q, rows_q, k_out, k, rows_k, Dh, wq, bq, wk, bk, eps, dtype, flags);
}

adaln_status adaln_qk_head_layernorm(void *q_out, const void *q, int64_t rows_q, void *k_out, const void *k,
                                     int64_t rows_k, int64_t Dh, const void *wq, const void *bq,
                                     const void *wk, const void *bk, float eps, int dtype, uint32_t flags,
                                     void *stream) {
    adaln_status st = check_qk(q_out, q, rows_q, k_out, k, rows_k, Dh, wq, bq, wk, bk, eps, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    QkArgs a{q_out, q, rows_q, k_out, k, rows_k, Dh, wq, bq, wk, bk, eps};
    return finish_launch(
        launch_qk_head_layernorm(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_qk_rmsnorm(const void *q_out, const void *q, int64_t rows_q, const void *k_out,
                                  const void *k, int64_t rows_k, int64_t Dh, const void *wq, const void *wk,
                                  float eps, int dtype, uint32_t flags) {
    return check_qk(q_out, q, rows_q, k_out, k, rows_k, Dh, wq, wq, wk, wk, eps, dtype, flags);
}

adaln_status adaln_qk_rmsnorm(void *q_out, const void *q, int64_t rows_q, void *k_out, const void *k,
                              int64_t rows_k, int64_t Dh, const void *wq, const void *wk, float eps, int dtype,
                              uint32_t flags, void *stream) {
    adaln_status st = check_qk(q_out, q, rows_q, k_out, k, rows_k, Dh, wq, wq, wk, wk, eps, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    QkArgs a{q_out, q, rows_q, k_out, k, rows_k, Dh, wq, nullptr, wk, nullptr, eps, true};
    return finish_launch(
        launch_qk_head_layernorm(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_ln_modulate_fp8(const void *out, const void *qscale, const void *x, int64_t B, int64_t N,
                                      int64_t D, int64_t sxB, int64_t sxN, int64_t sxD, const void *scale,
                                      int64_t s_scale_b, const void *shift, int64_t s_shift_b, float eps, int dtype,
                                      uint32_t flags) {
    return check_ln_fp8(out, qscale, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps, dtype,
                        flags);
}

int adaln_ln_modulate_fp8_variant(const void *out, const void *qscale, const void *x, int64_t B, int64_t N, int64_t D,
                                  int64_t sxB, int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b,
                                  const void *shift, int64_t s_shift_b, float eps, int dtype, uint32_t flags) {
    adaln_status st = check_ln_fp8(out, qscale, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps,
                                   dtype, flags);
    if (st != ADALN_OK) return -(int)st;
    LnArgs a{(void *)out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps};
    a.qscale = (const float *)qscale;
    return ln_modulate_path(a);
}

adaln_status adaln_ln_modulate_fp8(void *out, const void *qscale, const void *x, int64_t B, int64_t N, int64_t D,
                                  int64_t sxB, int64_t sxN, int64_t sxD, const void *scale, int64_t s_scale_b,
                                  const void *shift, int64_t s_shift_b, float eps, int dtype, uint32_t flags,
                                  void *stream) {
    adaln_status st = check_ln_fp8(out, qscale, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps,
                                   dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    LnArgs a{out, x, B, N, D, sxB, sxN, sxD, scale, s_scale_b, shift, s_shift_b, eps};
    a.qscale = (const float *)qscale;
    return finish_launch(launch_norm_scale_shift(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_temb_table_slices(const void *out, int64_t s_out_k, const void *table, int table_dtype,
                                        const void *temb, int temb_dtype, int64_t B, int64_t S, int64_t K,
                                        int64_t D, uint32_t flags) {
    return check_temb(out, s_out_k, table, table_dtype, temb, temb_dtype, B, S, K, D, flags);
}

adaln_status adaln_temb_table_slices(void *out, int64_t s_out_k, const void *table, int table_dtype,
                                    const void *temb, int temb_dtype, int64_t B, int64_t S, int64_t K, int64_t D,
                                    uint32_t flags, void *stream) {
    adaln_status st = check_temb(out, s_out_k, table, table_dtype, temb, temb_dtype, B, S, K, D, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    TembArgs a{out, K > 1 ? s_out_k : B * S * D, table, table_dtype, temb, temb_dtype, B, S, K, D};
    return finish_launch(launch_temb_table_slices(a, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_residual_gate_add(const void *out, const void *x, const void *gate, int64_t s_gate_b,
                                         const void *y, int64_t B, int64_t N, int64_t D, int dtype,
                                         uint32_t flags) {
    return check_gate(out, x, gate, s_gate_b, y, B, N, D, dtype, flags);
}

adaln_status adaln_residual_gate_add(void *out, const void *x, const void *gate, int64_t s_gate_b,
                                     const void *y, int64_t B, int64_t N, int64_t D, int dtype,
                                     uint32_t flags, void *stream) {
    adaln_status st = check_gate(out, x, gate, s_gate_b, y, B, N, D, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    GateArgs a{out, x, gate, s_gate_b, y, B, N, D};
    return finish_launch(
        launch_residual_gate_add(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

adaln_status adaln_can_bias_gelu_tanh(const void *out, const void *x, const void *bias, int64_t rows,
                                      int64_t width, int dtype, uint32_t flags) {
    return check_gelu(out, x, bias, rows, width, dtype, flags);
}

adaln_status adaln_bias_gelu_tanh(void *out, const void *x, const void *bias, int64_t rows, int64_t width,
                                  int dtype, uint32_t flags, void *stream) {
    adaln_status st = check_gelu(out, x, bias, rows, width, dtype, flags);
    if (st != ADALN_OK) return st;
    int dev;
    DeviceInfo info;
    if ((st = current_device(&dev)) != ADALN_OK || (st = device_info(dev, &info)) != ADALN_OK) return st;
    const void *table = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_dev[dev].gelu) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            cudaError_t e = cudaStreamIsCapturing((cudaStream_t)stream, &cs);
            if (e != cudaSuccess) return cuda_fail(e);
            if (cs != cudaStreamCaptureStatusNone) {
                snprintf(g_err, sizeof(g_err),
                         "GELU tables not built on device %d: call adaln_init before stream capture", dev);
                return ADALN_E_CUDA;
            }
            if ((st = build_tables_locked(dev)) != ADALN_OK) return st;
        }
        table = (const uint16_t *)g_dev[dev].gelu + (dtype == ADALN_FP16 ? 65536 : 0);
    }
    GeluArgs a{out, x, bias, rows, width, table};
    return finish_launch(
        launch_bias_gelu_tanh(a, dtype, (flags & ADALN_FLAG_PDL) != 0, (cudaStream_t)stream, info));
}

}  // extern "C"
