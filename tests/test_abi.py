"""The C-ABI library: it builds, loads, exports every symbol include/sp24.h declares, and
its host-side argument checks reject bad calls before anything is enqueued.  Nothing
here launches a kernel (fake pointers are only ever used in calls that must fail
validation first)."""
import ctypes
import os
import re

import pytest
import torch

import structured_sparse_matrix_gb300 as sp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sp24.h")

OK, INVALID, UNSUPPORTED, ALIGN, CUDA, TIMEOUT, NOT24, NODEV = range(8)
F16, BF16, E4M3, E5M2, S8, U8, F32, S32 = range(8)
FAKE = ctypes.c_void_p(0x10000)       # 16-byte aligned, never dereferenced
FAKE_ODD = ctypes.c_void_p(0x10008)   # 8-byte aligned only


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sp24_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("sp24_compress", "sp24_decompress", "sp24_meta_bytes", "sp24_meta_prepare",
              "sp24_mma", "sp24_status_string", "sp24_version"):
        assert n in names
    assert set(names) == set(sp.EXPORTS)


def test_library_exports_every_declared_symbol():
    L = sp.lib()
    for name in declared_functions():
        assert hasattr(L, name), name


def declared_arity():
    """Number of parameters of every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(sp24_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_argument_lists_match_the_header():
    L = sp.lib()
    arity = declared_arity()
    assert set(arity) == set(declared_functions())
    for name, n in arity.items():
        argtypes = getattr(L, name).argtypes
        if argtypes is not None:  # functions called without arguments have none set
            assert len(argtypes) == n, (name, len(argtypes), n)
        else:
            assert n == 0, name


def test_version_and_status_strings():
    L = sp.lib()
    assert L.sp24_version() == 1
    for code in range(8):
        s = L.sp24_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert L.sp24_status_string(99) == b"unknown status"


def test_meta_bytes_host_only():
    L = sp.lib()
    # per (128-row tile, stage) one [128 lanes][W words] block: W = 4 (2 KiB) for 16-bit
    # types with 128 dense K per stage, W = 8 (4 KiB) for FP8 with 256; M rounds up to
    # 256 rows, so for whole tiles and stages the image is M x K / 8 bytes
    assert L.sp24_meta_bytes(BF16, 4096, 4096) == 32 * 32 * 2048 == 4096 * 4096 // 8
    assert L.sp24_meta_bytes(F16, 64, 128) == 2 * 2048
    assert L.sp24_meta_bytes(F16, 129, 160) == 2 * 2 * 2048
    assert L.sp24_meta_bytes(E4M3, 8192, 8192) == 64 * 32 * 4096 == 8192 * 8192 // 8
    # 8-bit integers use the 16-bit layout (their product runs on the bf16 path)
    assert L.sp24_meta_bytes(S8, 8192, 8192) == 64 * 64 * 2048
    assert L.sp24_meta_bytes(F16, 64, 100) == 0      # K % 32 != 0
    assert L.sp24_meta_bytes(F32, 64, 128) == 0      # not an operand type


def _compress(t=F16, M=64, K=128, A=FAKE, lda=128, mask=None, ldm=128, mode=0, values=FAKE,
              ldv=64, index=FAKE, ldi=4):
    return sp.lib().sp24_compress(t, M, K, A, lda, mask, ldm, mode, values, ldv, index, ldi,
                                  None, None)


def test_compress_argument_checks():
    assert _compress(t=F32) == UNSUPPORTED
    assert _compress(mode=7) == INVALID
    assert _compress(K=100) == INVALID
    assert _compress(M=-1) == INVALID
    assert _compress(A=None) == INVALID
    assert _compress(mode=1, mask=None) == INVALID
    assert _compress(lda=64) == INVALID
    assert _compress(ldv=32) == INVALID
    assert _compress(ldi=2) == INVALID
    assert _compress(A=FAKE_ODD) == ALIGN
    assert _compress(lda=132) == ALIGN          # 264-byte pitch
    assert _compress(M=0) == OK                 # nothing to do, nothing enqueued
    assert _compress(K=0) == OK


def _mma(ta=BF16, tb=BF16, tc=F32, td=F32, M=128, N=128, K=128, values=FAKE, ldv=64, meta=FAKE,
         B=FAKE, ldb=128, C=FAKE, ldc=128, D=FAKE, ldd=128, ws=None, ws_bytes=0):
    return sp.lib().sp24_mma(ta, tb, tc, td, M, N, K, values, ldv, meta, B, ldb, C, ldc, D, ldd,
                             ws, ws_bytes, None, None)


def test_mma_argument_checks():
    assert _mma(ta=F16, tb=BF16) == UNSUPPORTED
    assert _mma(ta=E4M3, tb=BF16) == UNSUPPORTED
    assert _mma(ta=BF16, tb=E4M3) == UNSUPPORTED
    assert _mma(td=S32) == UNSUPPORTED
    assert _mma(tc=S32) == UNSUPPORTED
    assert _mma(ta=F32, tb=F32) == UNSUPPORTED
    assert _mma(ta=S8, tb=U8, tc=S32, td=S32) == UNSUPPORTED      # B must be signed
    assert _mma(ta=U8, tb=S8, tc=S32, td=F32) == UNSUPPORTED      # integers give s32
    assert _mma(ta=S8, tb=S8, tc=F32, td=S32) == UNSUPPORTED      # C must be s32
    # integer operands need the workspace
    assert _mma(ta=S8, tb=S8, tc=S32, td=S32) == INVALID
    need = sp.lib().sp24_mma_workspace_bytes(S8, S8, 128, 128, 128)
    assert need == 128 * 64 * 2 + 128 * 128 * 2
    assert _mma(ta=S8, tb=S8, tc=S32, td=S32, ws=FAKE, ws_bytes=need - 16) == INVALID
    assert _mma(ta=S8, tb=S8, tc=S32, td=S32, ws=FAKE_ODD, ws_bytes=need) == ALIGN
    assert sp.lib().sp24_mma_workspace_bytes(BF16, BF16, 128, 128, 128) == 0
    assert _mma(K=48) == INVALID
    assert _mma(N=-3) == INVALID
    assert _mma(D=None) == INVALID
    assert _mma(B=None) == INVALID
    assert _mma(ldb=64) == INVALID
    assert _mma(ldd=100) == INVALID
    assert _mma(ldc=100) == INVALID
    assert _mma(D=FAKE_ODD) == ALIGN
    assert _mma(B=FAKE_ODD) == ALIGN
    assert _mma(ldd=130) == ALIGN               # 520-byte pitch
    assert _mma(M=0) == OK
    assert _mma(N=0) == OK
    assert _mma(meta=None) == INVALID          # sp24_mma needs the image
    assert _mma(meta=FAKE_ODD) == ALIGN


def _mma_index(ta=BF16, tb=BF16, tc=F32, td=F32, M=128, N=128, K=128, values=FAKE, ldv=64,
               index=FAKE, ldi=4, B=FAKE, ldb=128, C=FAKE, ldc=128, D=FAKE, ldd=128, ws=None,
               ws_bytes=0):
    return sp.lib().sp24_mma_index(ta, tb, tc, td, M, N, K, values, ldv, index, ldi, B, ldb, C,
                                   ldc, D, ldd, ws, ws_bytes, None, None)


def test_mma_index_argument_checks():
    # the same type and shape rules as sp24_mma
    assert _mma_index(ta=F16, tb=BF16) == UNSUPPORTED
    assert _mma_index(ta=F32, tb=F32) == UNSUPPORTED
    assert _mma_index(ta=S8, tb=S8, tc=S32, td=S32) == INVALID        # no workspace
    assert _mma_index(K=48) == INVALID
    assert _mma_index(D=None) == INVALID
    # the canonical index: present, ldi >= K/32 words, 4-byte aligned, any pitch
    assert _mma_index(index=None) == INVALID
    assert _mma_index(ldi=3) == INVALID
    assert _mma_index(index=ctypes.c_void_p(0x10002)) == ALIGN
    assert _mma_index(B=FAKE_ODD) == ALIGN
    assert _mma_index(M=0) == OK


def _bmma(ta=BF16, tb=BF16, tc=F32, td=F32, batch=3, M=128, N=128, K=128, sv=None, sm=None,
          sb=None, sc=None, sd=None, C=FAKE, D=FAKE):
    M_, N_, K_ = M, N, K
    sv = M_ * K_ // 2 if sv is None else sv
    sm = sp.lib().sp24_meta_bytes(ta, M_, K_) if sm is None else sm
    sb = K_ * N_ if sb is None else sb
    sc = M_ * N_ if sc is None else sc
    sd = M_ * N_ if sd is None else sd
    return sp.lib().sp24_mma_strided_batched(ta, tb, tc, td, batch, M, N, K, FAKE, K // 2, sv,
                                             FAKE, sm, FAKE, N, sb, C, N, sc, D, N, sd, None,
                                             None)


def test_batched_argument_checks():
    assert _bmma(ta=S8, tb=S8, tc=S32, td=S32) == UNSUPPORTED   # float operands only
    assert _bmma(ta=F16, tb=BF16) == UNSUPPORTED
    assert _bmma(batch=-1) == INVALID
    assert _bmma(batch=0) == OK                                   # nothing to do
    assert _bmma(sd=128 * 128 - 4) == INVALID                     # D blocks overlap
    assert _bmma(sm=1024) == INVALID                              # smaller than one image
    assert _bmma(sv=128 * 64 + 4) == ALIGN                        # 8200-byte stride
    assert _bmma(sd=128 * 128 + 2) == ALIGN
    assert _bmma(D=None) == INVALID


def test_meta_prepare_argument_checks():
    L = sp.lib()
    assert L.sp24_meta_prepare(F32, 64, 128, FAKE, 4, FAKE, None) == UNSUPPORTED
    assert L.sp24_meta_prepare(F16, 64, 100, FAKE, 4, FAKE, None) == INVALID
    assert L.sp24_meta_prepare(F16, 64, 128, FAKE, 2, FAKE, None) == INVALID
    assert L.sp24_meta_prepare(F16, 64, 128, FAKE, 4, FAKE_ODD, None) == ALIGN


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_no_device_means_no_cpu_fallback():
    # valid-looking arguments reach the device check and are refused: no CPU path exists
    assert _compress() == NODEV
    assert _mma() == NODEV
    assert _mma_index() == NODEV
    assert _mma_index(index=FAKE_ODD, ldi=6) == NODEV  # any 4-byte aligned index and pitch
    assert sp.lib().sp24_diag_wait_timeout(FAKE, 1000, None) == NODEV
    assert sp.lib().sp24_diag_mma_stall(BF16, 256, 256, 256, FAKE, 128, FAKE, FAKE, 256, FAKE,
                                        256, 1000, FAKE, None) == NODEV


S4, U4 = 8, 9


def test_four_bit_argument_checks():
    L = sp.lib()
    # the 16-bit metadata layout (the product runs widened to bf16)
    assert L.sp24_meta_bytes(S4, 4096, 4096) == L.sp24_meta_bytes(BF16, 4096, 4096)
    assert L.sp24_meta_bytes(U4, 129, 160) == 2 * 2 * 2048
    # pitches count elements: lda = 144 is 72 bytes, ldv = 80 is 40 bytes
    assert _compress(t=S4, lda=144) == ALIGN
    assert _compress(t=U4, ldv=80) == ALIGN
    assert _compress(t=S4, ldv=48) == INVALID
    assert _compress(t=U4, M=0) == OK
    assert L.sp24_decompress(S4, 64, 128, FAKE, 80, FAKE, 4, FAKE, 128, None) == ALIGN
    # products: both operands 4-bit (any sign mix), integer C and D
    assert _mma(ta=S4, tb=S8, tc=S32, td=S32) == UNSUPPORTED
    assert _mma(ta=S8, tb=S4, tc=S32, td=S32) == UNSUPPORTED
    assert _mma(ta=U4, tb=U4, tc=S32, td=F32) == UNSUPPORTED
    assert _mma(ta=S4, tb=U4, tc=F32, td=S32) == UNSUPPORTED
    need = L.sp24_mma_workspace_bytes(S4, U4, 128, 128, 128)
    assert need == L.sp24_mma_workspace_bytes(S8, S8, 128, 128, 128)
    assert L.sp24_mma_workspace_bytes(S4, S8, 128, 128, 128) == 0
    assert _mma(ta=S4, tb=U4, tc=S32, td=S32) == INVALID           # needs the workspace
    assert _mma(ta=U4, tb=S4, tc=S32, td=S32, ws=FAKE, ws_bytes=need, ldb=144) == ALIGN
    assert _mma(ta=U4, tb=S4, tc=S32, td=S32, ws=FAKE, ws_bytes=need, ldv=80) == ALIGN
    assert _bmma(ta=S4, tb=S4, tc=S32, td=S32) == UNSUPPORTED


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_four_bit_valid_calls_reach_the_device_check():
    need = sp.lib().sp24_mma_workspace_bytes(S4, S4, 128, 128, 128)
    assert _compress(t=S4) == NODEV
    assert _mma(ta=S4, tb=S4, tc=S32, td=S32, ws=FAKE, ws_bytes=need) == NODEV


def test_16bit_accumulator_argument_checks():
    assert _mma(tc=S32) == UNSUPPORTED
    assert _mma(td=S32) == UNSUPPORTED
    assert _mma(td=E4M3) == UNSUPPORTED
    assert _mma(tc=F16, ldc=132) == ALIGN          # 264-byte pitch
    assert _mma(tc=BF16, ldc=100) == INVALID
    assert _bmma(tc=F16, sc=128 * 128 + 4) == ALIGN  # 32776-byte stride


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device answer")
def test_16bit_accumulator_calls_reach_the_device_check():
    assert _mma(ta=F16, tb=F16, tc=F16, td=F16, ldc=136, ldd=136) == NODEV
    assert _mma(ta=BF16, tb=BF16, tc=BF16, td=BF16) == NODEV
    assert _mma(ta=E4M3, tb=E5M2, tc=BF16, td=F16) == NODEV


def test_compress_meta_argument_checks():
    L = sp.lib()

    def cm(t=F16, M=64, K=128, A=FAKE, lda=128, mask=None, ldm=128, mode=0, values=FAKE,
           ldv=64, index=FAKE, ldi=4, meta=FAKE):
        return L.sp24_compress_meta(t, M, K, A, lda, mask, ldm, mode, values, ldv, index, ldi,
                                    meta, None, None)
    assert cm(t=F32) == UNSUPPORTED
    assert cm(K=100) == INVALID
    assert cm(meta=None) == INVALID
    assert cm(mode=1) == INVALID                       # mask mode without a mask
    assert cm(ldi=2) == INVALID
    assert cm(meta=FAKE_ODD) == ALIGN
    assert cm(lda=132) == ALIGN
    assert cm(M=0) == OK
    if not torch.cuda.is_available():
        assert cm(index=None, ldi=0) == NODEV           # the index is optional
        assert cm() == NODEV


def test_grouped_argument_checks():
    L = sp.lib()

    def grouped(ta=BF16, tb=BF16, tc=F32, td=F32, probs=None, count=None):
        probs = probs if probs is not None else [dict()]
        arr = (sp.Problem * len(probs))()
        for i, d in enumerate(probs):
            f = dict(M=128, N=128, K=128, values=0x10000, ldv=64, meta=0x10000, B=0x10000,
                     ldb=128, C=0, ldc=128, D=0x10000, ldd=128)
            f.update(d)
            arr[i] = sp.Problem(**f)
        return L.sp24_mma_grouped(ta, tb, tc, td, arr, len(probs) if count is None else count,
                                  None, None)
    assert grouped(ta=S8, tb=S8, tc=S32, td=S32) == UNSUPPORTED
    assert grouped(ta=F16, tb=BF16) == UNSUPPORTED
    assert grouped(td=S32) == UNSUPPORTED
    assert grouped(count=-1) == INVALID
    assert grouped(count=0) == OK
    assert grouped(probs=[dict(K=48)]) == INVALID
    assert grouped(probs=[dict(), dict(D=0)]) == INVALID           # any bad problem refuses
    assert grouped(probs=[dict(ldb=132)]) == ALIGN
    assert grouped(probs=[dict(M=0), dict(N=0)]) == OK              # nothing to do
    if not torch.cuda.is_available():
        assert grouped(probs=[dict(), dict(M=300, N=40)]) == NODEV


def test_header_is_plain_c_and_cpp(tmp_path):
    # the boundary header compiles on its own as C99 and as C++17 (no torch or CUDA types)
    import shutil
    import subprocess
    for compiler, std, lang in (("gcc", "-std=c99", "c"), ("g++", "-std=c++17", "c++")):
        if shutil.which(compiler) is None:
            pytest.skip(f"{compiler} not available")
        r = subprocess.run([compiler, std, "-Wall", "-Wextra", "-pedantic", "-fsyntax-only",
                            "-x", lang, HEADER], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_gemm_give_up_self_test_validates_before_the_device():
    L = sp.lib()
    args = (256, 256, 256, FAKE, 128, FAKE, FAKE, 256, FAKE, 256)
    assert L.sp24_diag_mma_stall(S8, *args, 1000, FAKE, None) == UNSUPPORTED  # float only
    assert L.sp24_diag_mma_stall(BF16, *args, 0, FAKE, None) == INVALID       # no limit
    assert L.sp24_diag_mma_stall(BF16, *args, 2_000_000_000, FAKE, None) == INVALID
    assert L.sp24_diag_mma_stall(BF16, *args, 1000, None, None) == INVALID    # no status word
    assert L.sp24_diag_mma_stall(BF16, 256, 256, 100, *args[3:], 1000, FAKE, None) == INVALID


def test_sparse_matrix_state_round_trip():
    # a compressed operand saved with torch.save and loaded back is the same operand
    import io
    g = torch.Generator().manual_seed(3)
    values = torch.randn(64, 96, generator=g).to(torch.bfloat16)
    index = torch.randint(0, 2**31 - 1, (64, 6), generator=g, dtype=torch.int32)
    meta = torch.randint(0, 256, (64 * 6 * 4,), generator=g, dtype=torch.uint8)
    W = sp.SparseMatrix(values, index, meta, 192)
    buf = io.BytesIO()
    torch.save(W.state_dict(), buf)
    buf.seek(0)
    R = sp.SparseMatrix.from_state_dict(torch.load(buf))
    assert R.shape == W.shape == (64, 192)
    for a, b in ((R.values, values), (R.index, index), (R.meta, meta)):
        assert a.dtype == b.dtype and torch.equal(a, b)
