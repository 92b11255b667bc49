"""Host-side checks of the C ABI (no GPU): the library builds and loads,
exports every function ``include/fp8fg.h`` declares, and rejects bad
arguments before touching the device."""
import ctypes
import os
import re

import pytest

import fp8_fine_grained_gb300 as fg
from fp8_fine_grained_gb300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8fg.h")

EINVAL, EALIGN, EUNSUPPORTED = 1, 2, 3


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return fg.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"FP8FG_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)))


def test_header_declares_the_four_entry_points():
    names = declared_functions()
    for n in ("fp8_quant_1x128", "fp8_quant_128x128", "fp8_gemm_blockscaled", "fp8_grouped_gemm"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    raw = ctypes.CDLL(fg.LIB_PATH)
    for n in declared_functions():
        assert hasattr(raw, n), n


def test_status_strings(L):
    for code in range(7):
        assert fg.status_str(code).startswith("FP8FG")
    assert "unknown" in fg.status_str(99)


# Fake, never-dereferenced device addresses: validation must fail first.
A16 = ctypes.c_void_p(0x10000)
A8 = ctypes.c_void_p(0x10008)
NULL = None


def q1x128(L, **kw):
    a = dict(x=A16, rows=4, cols=256, ldx=256, q=A16, ldq=256, s=A16, lds=4, t=0)
    a.update(kw)
    return L.fp8_quant_1x128(a["x"], a["rows"], a["cols"], a["ldx"], a["q"], a["ldq"], a["s"], a["lds"], a["t"], NULL)


def test_quant_1x128_validation(L):
    assert q1x128(L, cols=200, ldx=200, ldq=200) == EINVAL          # cols % 128
    assert q1x128(L, rows=-1) == EINVAL
    assert q1x128(L, ldx=128) == EINVAL                              # ldx < cols
    assert q1x128(L, lds=2) == EINVAL                                # ld_s < rows
    assert q1x128(L, x=NULL) == EINVAL
    assert q1x128(L, x=A8) == EALIGN
    assert q1x128(L, ldx=260) == EALIGN
    assert q1x128(L, t=2) == EINVAL
    assert q1x128(L, t=1, rows=100) == EINVAL                        # transposed: rows % 128
    assert q1x128(L, rows=0) == 0                                    # empty: nothing launched
    assert q1x128(L) in (EUNSUPPORTED, 4)                            # valid args, no GPU here


def test_quant_128x128_validation(L):
    f = L.fp8_quant_128x128
    assert f(A16, 100, 128, 128, A16, 128, A16, NULL) == EINVAL
    assert f(A16, 128, 130, 130, A16, 130, A16, NULL) == EINVAL
    assert f(A8, 128, 128, 128, A16, 128, A16, NULL) == EALIGN
    assert f(A16, 0, 128, 128, A16, 128, A16, NULL) == 0


@pytest.mark.parametrize("entry", ["fp8_quant_128x128_dual", "fp8_quant_128x128_dual_pow2"])
def test_quant_128x128_dual_validation(L, entry):
    f = getattr(L, entry)
    # w, N, K, ldw, q, ldq, scales, qT, ldqT, scalesT
    assert f(A16, 100, 128, 128, A16, 128, A16, A16, 128, A16, NULL) == EINVAL    # N % 128
    assert f(A16, 128, 130, 130, A16, 130, A16, A16, 128, A16, NULL) == EINVAL    # K % 128
    assert f(A16, 256, 128, 128, A16, 128, A16, A16, 128, A16, NULL) == EINVAL    # ldqT < N
    assert f(A16, 128, 128, 128, A16, 128, A16, A8, 128, A16, NULL) == EALIGN     # qT
    assert f(A16, 128, 128, 128, A16, 128, A16, A16, 136, A16, NULL) == EALIGN    # ldqT % 16
    assert f(A16, 128, 128, 128, A16, 128, A16, NULL, 128, A16, NULL) == EINVAL   # missing qT
    assert f(A16, 0, 128, 128, A16, 128, A16, A16, 128, A16, NULL) == 0


def gemm(L, **kw):
    a = dict(mode=0, A=A16, sA=A16, lda=256, ldsa=128, B=A16, sB=A16, ldb=256, ldsb=2, M=128, N=256, K=256,
             C=A16, out=1, ldc=256)
    a.update(kw)
    return L.fp8_gemm_blockscaled(a["mode"], a["A"], a["sA"], a["lda"], a["ldsa"], a["B"], a["sB"], a["ldb"],
                                  a["ldsb"], a["M"], a["N"], a["K"], a["C"], a["out"], a["ldc"], NULL)


def test_gemm_validation(L):
    assert gemm(L, mode=3) == EINVAL
    assert gemm(L, out=2) == EINVAL
    assert gemm(L, K=0) == EINVAL
    assert gemm(L, K=200, lda=208, ldb=208) == EINVAL
    assert gemm(L, N=200, ldc=208) == EINVAL
    assert gemm(L, ldsa=100) == EINVAL                 # ld_sA < M
    assert gemm(L, ldsb=1) == EINVAL                   # fprop: ld_sB < K/128
    assert gemm(L, mode=2, ldsb=128) == EINVAL         # wgrad: ld_sB < N
    assert gemm(L, mode=1, ldb=128, ldsb=2) == EINVAL  # dgrad: ldb < N
    assert gemm(L, A=A8) == EALIGN
    assert gemm(L, lda=264) == EALIGN
    assert gemm(L, C=NULL) == EINVAL
    assert gemm(L, M=0) == 0
    assert gemm(L) in (EUNSUPPORTED, 4)


def test_grouped_validation(L):
    f = L.fp8_grouped_gemm

    def call(**kw):
        a = dict(X=A16, sX=A16, ldsx=64, T=64, ri=A16, off=A16, E=4, R=100, W=A16, sW=A16, N=256, K=256,
                 Y=A16, out=1, ldy=256)
        a.update(kw)
        return f(a["X"], a["sX"], a["ldsx"], a["T"], a["ri"], a["off"], a["E"], a["R"], a["W"], a["sW"], a["N"],
                 a["K"], a["Y"], a["out"], a["ldy"], NULL)

    assert call(E=0) == EINVAL
    assert call(E=5000) == EINVAL
    assert call(K=100) == EINVAL
    assert call(ldsx=32) == EINVAL
    assert call(off=NULL) == EINVAL
    assert call(X=A8) == EALIGN
    assert call(R=0) == 0
    assert call() in (EUNSUPPORTED, 4)


def test_quant_dual_validation(L):
    f = L.fp8_quant_1x128_dual
    ok = dict(x=A16, rows=256, cols=384, ldx=384, q=A16, ldq=384, s=A16, lds=256, qT=A16, ldqT=256, sT=A16,
              ldsT=384)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["x"], a["rows"], a["cols"], a["ldx"], a["q"], a["ldq"], a["s"], a["lds"], a["qT"], a["ldqT"],
                 a["sT"], a["ldsT"], NULL)

    assert call(rows=200, ldqT=200, lds=200) == EINVAL               # rows % 128
    assert call(cols=200, ldx=200, ldq=200, ldsT=200) == EINVAL      # cols % 128
    assert call(ldqT=128) == EINVAL                                   # ldqT < rows
    assert call(ldsT=256) == EINVAL                                   # ld_sT < cols
    assert call(qT=NULL) == EINVAL
    assert call(qT=A8) == EALIGN
    assert call(ldsT=386) == EALIGN
    assert call(rows=0) == 0
    assert call() in (EUNSUPPORTED, 4)


def test_quant_gather_validation(L):
    f = L.fp8_quant_1x128_gather
    ok = dict(x=A16, n_src=16, cols=256, ldx=256, ri=A16, rows=40, q=A16, ldq=256, s=A16, lds=40)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return f(a["x"], a["n_src"], a["cols"], a["ldx"], a["ri"], a["rows"], a["q"], a["ldq"], a["s"], a["lds"],
                 NULL)

    assert call(cols=200, ldx=200, ldq=200) == EINVAL
    assert call(lds=36) == EINVAL                                     # ld_s < rows
    assert call(ri=NULL) == EINVAL
    assert call(n_src=0) == EINVAL                                    # rows to read, no source rows
    assert call(x=A8) == EALIGN
    assert call(lds=42) == EALIGN
    assert call(rows=0) == 0
    assert call() in (EUNSUPPORTED, 4)


def test_grouped_without_row_index_needs_enough_rows(L):
    # rows already in expert order: row r of Xq feeds output row r, so the
    # row count may not exceed the rows Xq holds
    f = L.fp8_grouped_gemm

    def call(T, R):
        return f(A16, A16, 64, T, NULL, A16, 4, R, A16, A16, 256, 256, A16, 1, 256, NULL)

    assert call(T=60, R=64) == EINVAL
    assert call(T=64, R=64) in (EUNSUPPORTED, 4)


def test_gemm_e4m3_validation(L):
    f = L.fp8_gemm_blockscaled_e4m3

    def call(**kw):
        a = dict(mode=0, A=A16, sA=A16, lda=256, ldsa=128, B=A16, sB=A16, ldb=256, ldsb=2, M=128, N=256, K=256,
                 C=A16, ldc=256, sC=A16, ldsc=128)
        a.update(kw)
        return f(a["mode"], a["A"], a["sA"], a["lda"], a["ldsa"], a["B"], a["sB"], a["ldb"], a["ldsb"], a["M"],
                 a["N"], a["K"], a["C"], a["ldc"], a["sC"], a["ldsc"], NULL)

    assert call(mode=2) == EINVAL                      # wgrad output stays FP32
    assert call(ldsc=100) == EINVAL                    # ld_sC < M
    assert call(sC=NULL) == EINVAL
    assert call(sC=A8) == EALIGN
    assert call(ldsc=130) == EALIGN
    assert call(ldc=264) == EALIGN
    assert call(M=0) == 0
    assert call() in (EUNSUPPORTED, 4)


def test_pow2_quantisers_validate_like_their_counterparts(L):
    """The power-of-two entry points share the argument checks of the
    pages' quantisers: the same bad arguments give the same codes."""
    cases = [dict(), dict(cols=200, ldx=208, ldq=208), dict(lds=2), dict(t=2), dict(x=A8), dict(ldq=264),
             dict(rows=0), dict(t=1, rows=100)]
    for kw in cases:
        a = dict(x=A16, rows=4, cols=256, ldx=256, q=A16, ldq=256, s=A16, lds=4, t=0)
        a.update(kw)
        args = (a["x"], a["rows"], a["cols"], a["ldx"], a["q"], a["ldq"], a["s"], a["lds"], a["t"], NULL)
        assert L.fp8_quant_1x128_pow2(*args) == L.fp8_quant_1x128(*args), kw
    for kw in [dict(), dict(N=200), dict(K=100), dict(ldw=264), dict(w=A8), dict(N=0)]:
        a = dict(w=A16, N=256, K=256, ldw=256, q=A16, ldq=256, s=A16)
        a.update(kw)
        args = (a["w"], a["N"], a["K"], a["ldw"], a["q"], a["ldq"], a["s"], NULL)
        assert L.fp8_quant_128x128_pow2(*args) == L.fp8_quant_128x128(*args), kw
    dual = (A16, 256, 384, 384, A16, 384, A16, 256, A16, 256, A16, 384, NULL)
    assert L.fp8_quant_1x128_dual_pow2(*dual) == L.fp8_quant_1x128_dual(*dual)
    bad_dual = (A16, 200, 384, 384, A16, 384, A16, 256, A16, 256, A16, 384, NULL)
    assert L.fp8_quant_1x128_dual_pow2(*bad_dual) == EINVAL
    gat = (A16, 64, 256, 256, A16, 8, A16, 256, A16, 8, NULL)
    assert L.fp8_quant_1x128_gather_pow2(*gat) == L.fp8_quant_1x128_gather(*gat)
    assert L.fp8_quant_1x128_gather_pow2(A16, 64, 256, 256, NULL, 8, A16, 256, A16, 8, NULL) == EINVAL


def test_gemm_mx_validation(L):
    """fp8_gemm_mx takes fp8_gemm_blockscaled's arguments and checks them the
    same way."""
    cases = [dict(mode=3), dict(out=2), dict(K=0), dict(K=200, lda=208, ldb=208), dict(N=200, ldc=208),
             dict(ldsa=100), dict(ldsb=1), dict(mode=2, ldsb=128), dict(mode=1, ldb=128, ldsb=2), dict(A=A8),
             dict(lda=264), dict(C=NULL), dict(M=0), dict()]
    for kw in cases:
        a = dict(mode=0, A=A16, sA=A16, lda=256, ldsa=128, B=A16, sB=A16, ldb=256, ldsb=2, M=128, N=256, K=256,
                 C=A16, out=1, ldc=256)
        a.update(kw)
        args = (a["mode"], a["A"], a["sA"], a["lda"], a["ldsa"], a["B"], a["sB"], a["ldb"], a["ldsb"], a["M"],
                a["N"], a["K"], a["C"], a["out"], a["ldc"], NULL)
        assert L.fp8_gemm_mx(*args) == L.fp8_gemm_blockscaled(*args), kw


def test_grouped_gemm_mx_validation(L):
    f = L.fp8_grouped_gemm_mx

    def call(**kw):
        a = dict(X=A16, sX=A16, ldsx=100, off=A16, E=4, R=100, W=A16, sW=A16, N=256, K=256, Y=A16, out=1,
                 ldy=256)
        a.update(kw)
        return f(a["X"], a["sX"], a["ldsx"], a["off"], a["E"], a["R"], a["W"], a["sW"], a["N"], a["K"], a["Y"],
                 a["out"], a["ldy"], NULL)

    assert call(E=0) == EINVAL
    assert call(E=5000) == EINVAL
    assert call(K=100) == EINVAL
    assert call(N=200) == EINVAL
    assert call(out=2) == EINVAL
    assert call(ldsx=96) == EINVAL      # ld_sX < n_rows
    assert call(ldy=128) == EINVAL      # ldy < N
    assert call(off=NULL) == EINVAL
    assert call(X=A8) == EALIGN
    assert call(ldsx=102) == EALIGN
    assert call(R=0) == 0
    assert call(Y=NULL) == EINVAL
    assert call() in (EUNSUPPORTED, 4)


def test_quant_scatter_validation(L):
    f = L.fp8_quant_1x128_scatter

    def call(**kw):
        a = dict(x=A16, n=64, cols=256, ldx=256, d=A16, k=8, n_out=512, q=A16, ldq=256, s=A16, lds=512)
        a.update(kw)
        return f(a["x"], a["n"], a["cols"], a["ldx"], a["d"], a["k"], a["n_out"], a["q"], a["ldq"], a["s"],
                 a["lds"], NULL)

    assert call(k=0) == EINVAL
    assert call(k=17) == EINVAL
    assert call(cols=200, ldx=208, ldq=208) == EINVAL
    assert call(lds=500) == EINVAL      # ld_s < n_out
    assert call(d=NULL) == EINVAL
    assert call(x=A8) == EALIGN
    assert call(lds=514) == EALIGN
    assert call(n=0) == 0
    assert call(n_out=0, lds=0) == 0
    assert call() in (EUNSUPPORTED, 4)
    args = (A16, 64, 256, 256, A16, 8, 512, A16, 256, A16, 500, NULL)
    assert L.fp8_quant_1x128_scatter_pow2(*args) == f(*args) == EINVAL


def test_moe_combine_validation(L):
    f = L.fp8_moe_combine

    def call(**kw):
        a = dict(y=A16, ldy=256, rows=100, d=A16, w=A16, T=64, k=8, N=256, out=A16, kind=1, ldo=256)
        a.update(kw)
        return f(a["y"], a["ldy"], a["rows"], a["d"], a["w"], a["T"], a["k"], a["N"], a["out"], a["kind"],
                 a["ldo"], NULL)

    assert call(k=0) == EINVAL
    assert call(k=17) == EINVAL
    assert call(N=100, ldy=104, ldo=104) == EINVAL   # N % 8 != 0
    assert call(ldy=248) == EINVAL                   # ldy < N
    assert call(ldo=248) == EINVAL                   # ldo < N
    assert call(kind=2) == EINVAL
    assert call(d=NULL) == EINVAL
    assert call(y=A8) == EALIGN
    assert call(ldy=260) == EALIGN                   # rows not 16-byte aligned
    assert call(T=0) == 0
    assert call(N=0, ldy=0, ldo=0) == 0
    assert call() in (EUNSUPPORTED, 4)


def test_grouped_schedule_validation(L):
    f = L.fp8fg_set_grouped_schedule
    assert f(-1, 100) == EINVAL
    assert f(33, 100) == EINVAL                      # skinny tiles hold 32 token rows
    assert f(32, 0) == EINVAL
    assert f(32, 1001) == EINVAL
    try:
        assert f(0, 1) == 0
        assert f(16, 1000) == 0
        with pytest.raises(fg.Fp8fgError):
            fg.set_grouped_schedule(40)
    finally:
        assert f(32, 100) == 0                       # the defaults
