"""The C ABI without a GPU: the library loads, exports every function that
include/adaln.h declares, and validates arguments on the host (returning a
status and launching nothing) before making any CUDA call."""
import ctypes

import pytest


@pytest.fixture(scope="module")
def ad():
    import __graft_entry__
    __graft_entry__.build()
    import adaln_modulate_gb300
    return adaln_modulate_gb300


def test_every_declared_symbol_is_exported(ad):
    names = ad.header_functions()
    assert len(names) >= 14
    lib = ctypes.CDLL(ad.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    for n in names:
        assert hasattr(ad.capi, n), n


def test_status_strings(ad):
    for code in range(9):
        assert ad.capi.adaln_status_str(code).decode().startswith(ad.STATUS[code])
    assert b"unknown" in ad.capi.adaln_status_str(99)
    assert ad.capi.adaln_version() == 10000


# Fake but aligned "device" addresses: validation never dereferences them.
OUT, X, SC, SH = 0x10000000, 0x20000000, 0x30000000, 0x30100000


def ln_can(ad, out=OUT, x=X, B=2, N=16, D=2240, strides=None, sc=SC, ssb=6 * 2240, sh=SH,
           shb=6 * 2240, eps=1e-6, dtype=0, flags=0):
    strides = strides or (N * D, D, 1)
    return ad.capi.adaln_can_ln_modulate(out, x, B, N, D, *strides, sc, ssb, sh, shb, eps, dtype, flags)


def test_ln_validation(ad):
    assert ln_can(ad) == 0
    assert ln_can(ad, dtype=2) == 2
    assert ln_can(ad, x=None) == 1 and ln_can(ad, sc=None) == 1
    for D in (0, 2, 6, 65540):
        assert ln_can(ad, D=D) == 3, D
    assert ln_can(ad, B=0) == 3 and ln_can(ad, N=0) == 3
    assert ln_can(ad, strides=(16 * 2240, 2240, -1)) == 5
    assert ln_can(ad, ssb=-1) == 5
    assert ln_can(ad, eps=-1.0) == 6 and ln_can(ad, eps=float("inf")) == 6
    assert ln_can(ad, eps=float("nan")) == 6
    assert ln_can(ad, flags=2) == 6
    assert ln_can(ad, x=X + 1) == 4
    # out overlapping a non-contiguous x, or the scale rows, is refused
    assert ln_can(ad, out=X, strides=(2240 * 16, 1, 16)) == 7
    assert ln_can(ad, out=SC - 100) == 7
    # in place on contiguous x is allowed
    assert ln_can(ad, out=X) == 0


def test_ln_invalid_call_returns_before_cuda(ad):
    # status is returned from validation; no stream or device is touched
    st = ad.capi.adaln_ln_modulate(OUT, X, 2, 16, 6, 16 * 6, 6, 1, SC, 6, SH, 6, 1e-6, 0, 0, None)
    assert st == 3


def test_ln_path_selection(ad):
    v = ad.capi.adaln_ln_modulate_variant
    # GLM contiguous rows
    assert v(OUT, X, 1, 4096, 4096, 4096 * 4096, 4096, 1, SC, 4096, SH, 4096, 1e-5, 0, 0) == 0
    # Sana transposed view of (2, 2240, 1024), nmod = 6 chunks
    assert v(OUT, X, 2, 1024, 2240, 2240 * 1024, 1, 1024, SC + 2 * 2240, 6 * 2240, SC, 6 * 2240,
             1e-6, 0, 0) == 1
    # D too large for the register / shared-memory kernels, odd strides
    assert v(OUT, X, 1, 8, 8192, 8 * 8192, 8192, 1, SC, 8192, SH, 8192, 1e-5, 0, 0) == 2
    assert v(OUT, X, 1, 8, 512, 3 * 8 * 512, 3 * 512, 3, SC, 512, SH, 512, 1e-5, 0, 0) == 2
    # misaligned row pitch for 8-byte accesses
    assert v(OUT, X + 2, 1, 8, 512, 8 * 512, 512, 1, SC, 512, SH, 512, 1e-5, 0, 0) == 2
    assert v(OUT, X, 1, 8, 6, 48, 6, 1, SC, 6, SH, 6, 1e-5, 0, 0) == -3


def test_qk_validation(ad):
    c = ad.capi.adaln_can_qk_head_layernorm
    W = [0x40000000 + 0x1000 * i for i in range(4)]
    ok = lambda **kw: c(kw.get("qo", OUT), kw.get("q", X), kw.get("rq", 100), kw.get("ko", OUT + 0x100000),
                        kw.get("k", X + 0x100000), kw.get("rk", 100), kw.get("Dh", 128), *W,
                        kw.get("eps", 1e-6), kw.get("dtype", 0), 0)
    assert ok() == 0
    assert ok(Dh=132) == 3 and ok(Dh=2) == 3 and ok(Dh=66) == 3
    assert ok(rq=0, rk=0) == 3
    assert ok(rq=0, q=None, qo=None) == 0
    assert ok(q=None) == 1
    assert ok(q=X + 2) == 4
    assert ok(qo=X) == 0                      # in place
    assert ok(qo=X + 64) == 7                 # partial overlap
    assert ok(ko=OUT + 128) == 7              # outputs overlap each other
    assert ok(dtype=5) == 2


def test_gate_and_gelu_validation(ad):
    g = ad.capi.adaln_can_residual_gate_add
    assert g(OUT, X, SC, 4096, SH, 1, 4096, 4096, 0, 0) == 0
    assert g(OUT, X, SC, 4096, SH, 1, 4096, 0, 0, 0) == 3
    assert g(OUT, X, SC, -1, SH, 1, 4096, 4096, 0, 0) == 5
    assert g(X, X, SC, 4096, SH, 1, 4096, 4096, 0, 0) == 0           # in place on x
    assert g(X + 2, X, SC, 4096, SH, 1, 4096, 4096, 0, 0) == 7
    assert g(OUT, X + 1, SC, 4096, SH, 1, 4096, 4096, 0, 0) == 4
    b = ad.capi.adaln_can_bias_gelu_tanh
    big_out, big_x = 1 << 40, 1 << 41          # 906 MB tensors far apart
    assert b(big_out, big_x, SC, 32760, 13824, 0, 0) == 0
    assert b(big_out, big_x, SC, 32760, 13824, 1, 0) == 0
    assert b(OUT, X, SC, 32760, 13824, 0, 0) == 7     # out would run into x
    assert b(OUT, X, SC, 0, 13824, 0, 0) == 3
    assert b(OUT, X, None, 10, 10, 0, 0) == 1
    assert b(OUT, X, OUT + 4, 10, 10, 0, 0) == 7
    assert b(OUT, X, SC, 10, 10, 3, 0) == 2


def test_residual_ln_validation(ad):
    f = ad.capi.adaln_can_residual_gate_ln_modulate
    R, O, Y = 1 << 36, 1 << 37, 1 << 38       # x, y, r, out far apart (33.5 MB each)
    G, S, H = 1 << 39, (1 << 39) + 16384, (1 << 39) + 32768
    args = lambda r=R, o=O, x=X, g=G, y=Y, D=4096, eps=1e-5, dt=0, fl=0: (
        r, o, x, g, 0, y, 1, 4096, D, S, 0, H, 0, eps, dt, fl)
    assert f(*args()) == 0
    assert f(*args(r=X)) == 0                   # in-place residual update on x
    assert f(*args(r=Y)) == 0                   # or on y
    assert f(*args(o=R)) == 7                   # out on r
    assert f(*args(o=X)) == 7                   # out on x
    assert f(*args(o=Y + 64)) == 7              # out into y
    assert f(*args(r=S - 8)) == 7               # r into the scale row
    assert f(*args(D=4098)) == 3                # D % 4 != 0
    assert f(*args(eps=-1.0)) == 6
    assert f(*args(dt=2)) == 2
    assert f(*args(fl=4)) == 6
    assert f(*args(g=0)) == 1
    assert f(*args(x=X + 1)) == 4               # odd address


def test_norm_scale_shift_validation(ad):
    f = ad.capi.adaln_can_norm_scale_shift
    R, O, Y = 1 << 36, 1 << 37, 1 << 38
    T = 1 << 39                                  # a per-token (B, N, 6, D) table
    B, N, D = 2, 64, 1024

    def args(norm=1, r=R, o=O, x=X, g=T, sgb=N * 6 * D, sgn=6 * D, sgd=1, y=Y, sc=T + 2 * D, ssn=6 * D,
             sh=T + 4 * D, eps=1e-6, dt=0, fl=0, strides=None):
        return (norm, r, o, x, B, N, D, *(strides or (N * D, D, 1)), g, sgb, sgn, sgd, y, sc, N * 6 * D, ssn,
                sh, N * 6 * D, ssn, eps, dt, fl)

    assert f(*args()) == 0
    assert f(*args(norm=0)) == 0
    assert f(*args(norm=2)) == 6                 # unknown norm
    assert f(*args(sgd=0, sgn=1, sgb=N, g=T)) == 0   # a per-token scalar gate
    assert f(*args(sgd=2)) == 5                  # gate element stride must be 0 or 1
    assert f(*args(y=0)) == 1 and f(*args(r=0)) == 1
    assert f(*args(strides=(N * D * 2, D * 2, 2))) == 5   # a gate needs contiguous x
    assert f(*args(r=X)) == 0 and f(*args(r=Y)) == 0      # in-place residual update
    assert f(*args(o=X)) == 7 and f(*args(o=R)) == 7
    assert f(*args(r=T + 64)) == 7               # r into the table
    assert f(*args(o=T + 2 * D + 6 * D * N + 8)) == 7     # out into a later token's scale row
    assert f(*args(ssn=-6 * D)) == 5
    # without a gate: any strides, y / r ignored, out == contiguous x allowed
    assert f(*args(g=0, y=0, r=0)) == 0
    assert f(*args(g=0, y=0, r=0, o=X)) == 0
    assert f(*args(g=0, y=0, r=0, strides=(N * D * 2, 1, N * 2))) == 0
    g = ad.capi.adaln_can_rmsnorm_scale_shift
    assert g(O, X, B, N, D, N * D, D, 1, T, 0, 0, T + 2 * D, 0, 0, 1e-6, 0, 0) == 0
    assert g(O, X, B, N, D, N * D, D, 1, T, 0, 0, T + 2 * D, 0, 0, float("nan"), 0, 0) == 6
    assert g(T + 2 * D, X, B, N, D, N * D, D, 1, T, 0, 0, T + 2 * D, 0, 0, 1e-6, 0, 0) == 7


def test_qk_rmsnorm_validation(ad):
    f = ad.capi.adaln_can_qk_rmsnorm
    Q, K, QO, KO, W = 1 << 36, 1 << 37, 1 << 38, 1 << 39, 1 << 40
    assert f(QO, Q, 100, KO, K, 100, 128, W, W + 256, 1e-6, 0, 0) == 0
    assert f(QO, Q, 100, None, None, 0, 128, W, None, 1e-6, 0, 0) == 0
    assert f(QO, Q, 100, KO, K, 100, 130, W, W + 256, 1e-6, 0, 0) == 3
    assert f(QO, Q, 100, KO, K, 100, 128, None, W, 1e-6, 0, 0) == 1
    assert f(QO, Q, 100, KO, K, 100, 128, W, W + 256, 1e-6, 0, 0) == 0
    assert f(W, Q, 100, KO, K, 100, 128, W, W + 256, 1e-6, 0, 0) == 7   # q_out on the weight
    assert f(QO, Q, 100, KO, K, 100, 128, W + 4, W + 256, 1e-6, 0, 0) == 4


def test_temb_table_slices_validation(ad):
    f = ad.capi.adaln_can_temb_table_slices
    O, T, E = 1 << 36, 1 << 37, 1 << 38
    B, S, K, D = 1, 100, 6, 3072
    ok = (O, B * S * D, T, 2, E, 0, B, S, K, D, 0)
    assert f(*ok) == 0
    a = list(ok)
    a[3] = 3
    assert f(*a) == 2                              # table dtype
    a = list(ok)
    a[5] = -1
    assert f(*a) == 2                              # temb dtype
    a = list(ok)
    a[1] = B * S * D - 8
    assert f(*a) == 5                              # slices would overlap
    a = list(ok)
    a[0] = O + 2
    assert f(*a) == 4                              # out not 4-byte aligned
    a = list(ok)
    a[0] = E + 64
    assert f(*a) == 7                              # out over temb
    a = list(ok)
    a[2] = O + 4 * (B * S * D * 5 + 8)
    assert f(*a) == 7                              # table inside the last slice
    a = list(ok)
    a[9] = 0
    assert f(*a) == 3
    a = list(ok)
    a[10] = 2
    assert f(*a) == 6
    assert f(O, 0, T, 0, E, 1, 2, 3, 1, 8, 0) == 0  # K = 1 ignores the slice stride


def test_ln_modulate_fp8_validation(ad):
    f = ad.capi.adaln_can_ln_modulate_fp8
    O, Q, X, S, H = 1 << 36, 1 << 37, 1 << 38, 1 << 39, (1 << 39) + 8192
    B, N, D = 1, 4608, 3072
    args = lambda o=O, q=Q, x=X, s=S, strides=None, eps=1e-6, dt=0, fl=0: (
        o, q, x, B, N, D, *(strides or (N * D, D, 1)), s, 0, H, 0, eps, dt, fl)
    assert f(*args()) == 0
    assert f(*args(q=0)) == 1
    assert f(*args(q=Q + 2)) == 4                 # the scale is a 4-byte float
    assert f(*args(o=X)) == 7                     # no in-place form
    assert f(*args(o=S - 100)) == 7
    assert f(*args(o=Q - 8)) == 7                 # out over the scale value
    assert f(*args(o=O + 1)) == 0                 # byte outputs need no alignment
    assert f(*args(dt=2)) == 2 and f(*args(eps=-1.0)) == 6 and f(*args(fl=8)) == 6
    assert f(*args(strides=(N * D, 1, N))) == 0   # any strides (the general kernel)


def test_huge_strides_are_refused(ad):
    # a stride past 2^46 elements would overflow the byte extents of the overlap checks
    big = 1 << 50
    assert ln_can(ad, strides=(big, 2240, 1)) == 5
    assert ln_can(ad, ssb=big) == 5
    f = ad.capi.adaln_can_norm_scale_shift
    assert f(0, 0, OUT, X, 2, 16, 2240, 16 * 2240, 2240, 1, 0, 0, 0, 1, 0, SC, 6 * 2240, big, SH, 6 * 2240, 0,
             1e-6, 0, 0) == 5
    assert ad.capi.adaln_can_residual_gate_add(OUT, X, SC, big, X + (1 << 30), 2, 16, 2240, 0, 0) == 5
