"""structured_sparse_matrix_gb300 -- 2:4 structured-sparse multiply-accumulate on GB300.

A thin ctypes binding over the C ABI of ``libsp24.so`` (``include/sp24.h``).  Every step
of the computation runs in the library's sm_103a kernels; this module only allocates the
output tensors with PyTorch, passes raw device pointers and the current CUDA stream, and
turns non-OK status codes into exceptions.  There is no CPU fallback: if the library is
missing or no sm_103 device is current, calls raise.

    values, index = compress(A, mode="mask", mask=keep)     # A: M x K on cuda
    meta = meta_prepare(index, A.dtype, M, K)
    D = mma(values, meta, B, C, out_dtype=torch.float32)     # D = A_sp @ B + C

4-bit integer operands ("s4", "u4") travel as uint8 tensors holding two elements per
byte (element 2i in the low nibble); the functions take them with ``elem="s4"`` (or
``a_elem`` / ``b_elem`` for ``mma``), and their shapes count bytes along the packed
dimension (A: M x K/2 bytes, values: M x K/4 bytes, B: K x N/2 bytes).
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import _build

__all__ = ["lib", "compress", "compress_meta", "decompress", "meta_bytes", "meta_prepare", "mma",
           "mma_index", "mma_batched", "mma_grouped",
           "workspace_bytes",
           "SparseMatrix", "Sp24Error", "DEV_NOT_2_4", "DEV_TIMEOUT", "DTYPE_CODES"]

DTYPE_CODES = {
    torch.float16: 0, torch.bfloat16: 1, torch.float8_e4m3fn: 2, torch.float8_e5m2: 3,
    torch.int8: 4, torch.uint8: 5, torch.float32: 6, torch.int32: 7,
}
# 4-bit types have no torch dtype: they are named by string
NAMED_CODES = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3, "s8": 4, "u8": 5, "f32": 6, "s32": 7,
               "s4": 8, "u4": 9}
PACKED4 = ("s4", "u4")
MODES = {"exact": 0, "mask": 1, "magnitude": 2}
DEV_NOT_2_4 = 1
DEV_TIMEOUT = 2

# every symbol include/sp24.h declares
EXPORTS = ("sp24_compress", "sp24_compress_meta", "sp24_decompress", "sp24_meta_bytes", "sp24_meta_prepare",
           "sp24_mma_workspace_bytes", "sp24_mma", "sp24_mma_index", "sp24_mma_strided_batched",
           "sp24_mma_grouped",
           "sp24_mma_i8_noalloc",
           "sp24_diag_wait_timeout", "sp24_diag_mma_stall", "sp24_status_string", "sp24_version")

class Problem(ctypes.Structure):
    """One problem of sp24_mma_grouped (the C struct sp24_mma_problem)."""
    _fields_ = [("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("values", ctypes.c_void_p), ("ldv", ctypes.c_int64),
                ("meta", ctypes.c_void_p),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("D", ctypes.c_void_p), ("ldd", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


class Sp24Error(RuntimeError):
    def __init__(self, fn: str, code: int, text: str):
        super().__init__(f"{fn} failed: {text} (status {code})")
        self.code = code


def lib():
    """Load libsp24.so (building it in-tree with nvcc if it is absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not _build.up_to_date():
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError("libsp24.so is missing and could not be built")
            L = ctypes.CDLL(path)
            i64, p, i32, u64 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64
            L.sp24_compress.restype = i32
            L.sp24_compress.argtypes = [i32, i64, i64, p, i64, p, i64, i32, p, i64, p, i64, p, p]
            L.sp24_compress_meta.restype = i32
            L.sp24_compress_meta.argtypes = [i32, i64, i64, p, i64, p, i64, i32, p, i64, p, i64,
                                             p, p, p]
            L.sp24_decompress.restype = i32
            L.sp24_decompress.argtypes = [i32, i64, i64, p, i64, p, i64, p, i64, p]
            L.sp24_meta_bytes.restype = ctypes.c_size_t
            L.sp24_meta_bytes.argtypes = [i32, i64, i64]
            L.sp24_meta_prepare.restype = i32
            L.sp24_meta_prepare.argtypes = [i32, i64, i64, p, i64, p, p]
            L.sp24_mma_workspace_bytes.restype = ctypes.c_size_t
            L.sp24_mma_workspace_bytes.argtypes = [i32, i32, i64, i64, i64]
            L.sp24_mma.restype = i32
            L.sp24_mma.argtypes = [i32, i32, i32, i32, i64, i64, i64, p, i64, p, p, i64, p, i64,
                                   p, i64, p, ctypes.c_size_t, p, p]
            L.sp24_mma_index.restype = i32
            L.sp24_mma_index.argtypes = [i32, i32, i32, i32, i64, i64, i64, p, i64, p, i64, p,
                                         i64, p, i64, p, i64, p, ctypes.c_size_t, p, p]
            L.sp24_mma_strided_batched.restype = i32
            L.sp24_mma_strided_batched.argtypes = [i32, i32, i32, i32, i64, i64, i64, i64, p, i64,
                                                   i64, p, i64, p, i64, i64, p, i64, i64, p,
                                                   i64, i64, p, p]
            L.sp24_mma_grouped.restype = i32
            L.sp24_mma_grouped.argtypes = [i32, i32, i32, i32, ctypes.POINTER(Problem), i64, p, p]
            L.sp24_mma_i8_noalloc.restype = i32
            L.sp24_mma_i8_noalloc.argtypes = [i32, i32, i32, i32, i64, i64, i64, p, i64, p, p,
                                              i64, p, i64, p, i64, p, p]
            L.sp24_diag_wait_timeout.restype = i32
            L.sp24_diag_wait_timeout.argtypes = [p, u64, p]
            L.sp24_diag_mma_stall.restype = i32
            L.sp24_diag_mma_stall.argtypes = [i32, i64, i64, i64, p, i64, p, p, i64, p, i64, u64,
                                              p, p]
            L.sp24_status_string.restype = ctypes.c_char_p
            L.sp24_status_string.argtypes = [i32]
            L.sp24_version.restype = i32
            _lib = L
    return _lib


def _check(fn: str, code: int):
    if code != 0:
        raise Sp24Error(fn, code, lib().sp24_status_string(code).decode())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _code(dtype):
    if isinstance(dtype, str):
        if dtype not in NAMED_CODES:
            raise TypeError(f"unsupported element type {dtype!r}")
        return NAMED_CODES[dtype]
    if dtype not in DTYPE_CODES:
        raise TypeError(f"unsupported element type {dtype}")
    return DTYPE_CODES[dtype]


def _ld(t, elem=None):
    """Leading dimension in elements (4-bit types: two per byte of a uint8 tensor)."""
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError("expected a 2-D row-major tensor (unit column stride)")
    return t.stride(0) * (2 if elem in PACKED4 else 1)


def _elem_code(t, elem):
    """Element code of tensor t, read as 4-bit elements when elem is "s4" / "u4"."""
    if elem is None:
        return _code(t.dtype)
    if elem not in PACKED4:
        raise ValueError(f"elem must be None, 's4' or 'u4', not {elem!r}")
    if t.dtype != torch.uint8:
        raise TypeError("4-bit operands travel as uint8 tensors (two elements per byte)")
    return _code(elem)


def compress(A: torch.Tensor, mode: str = "exact", mask: torch.Tensor | None = None,
             status: torch.Tensor | None = None, stream=None, elem: str | None = None):
    """Dense M x K (2:4 along K) -> (values M x K/2, index M x K/32 int32 words).

    elem="s4" / "u4": A is M x K/2 packed bytes and values M x K/4 packed bytes."""
    t = _elem_code(A, elem)
    per = 2 if elem in PACKED4 else 1
    M, K = A.shape[0], A.shape[1] * per
    vcols = K // 2 // per
    if per == 2:  # K/4 bytes a row: pad the pitch to 16 bytes (K = 32 gives 8)
        values = torch.empty((M, (vcols + 15) // 16 * 16), dtype=A.dtype,
                             device=A.device)[:, :vcols]
    else:
        values = torch.empty((M, vcols), dtype=A.dtype, device=A.device)
    index = torch.empty((M, K // 32), dtype=torch.int32, device=A.device)
    m = None
    ldm = K
    if mode == "mask":
        if mask is None:
            raise ValueError("mask mode needs a mask")
        m = mask.to(torch.uint8) if mask.dtype != torch.uint8 else mask
        ldm = _ld(m)
    _check("sp24_compress", lib().sp24_compress(
        t, M, K, _ptr(A), _ld(A, elem), _ptr(m), ldm, MODES[mode], _ptr(values),
        _ld(values, elem), _ptr(index), _ld(index), _ptr(status), _stream(stream)))
    return values, index


def compress_meta(A: torch.Tensor, mode: str = "exact", mask: torch.Tensor | None = None,
                  status: torch.Tensor | None = None, stream=None, elem: str | None = None,
                  with_index: bool = True):
    """compress() and meta_prepare() in one pass: (values, index or None, meta)."""
    t = _elem_code(A, elem)
    per = 2 if elem in PACKED4 else 1
    M, K = A.shape[0], A.shape[1] * per
    vcols = K // 2 // per
    if per == 2:
        values = torch.empty((M, (vcols + 15) // 16 * 16), dtype=A.dtype,
                             device=A.device)[:, :vcols]
    else:
        values = torch.empty((M, vcols), dtype=A.dtype, device=A.device)
    index = torch.empty((M, K // 32), dtype=torch.int32, device=A.device) if with_index else None
    nbytes = int(lib().sp24_meta_bytes(t, M, K))
    meta = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=A.device)
    m = None
    ldm = K
    if mode == "mask":
        if mask is None:
            raise ValueError("mask mode needs a mask")
        m = mask.to(torch.uint8) if mask.dtype != torch.uint8 else mask
        ldm = _ld(m)
    _check("sp24_compress_meta", lib().sp24_compress_meta(
        t, M, K, _ptr(A), _ld(A, elem), _ptr(m), ldm, MODES[mode], _ptr(values),
        _ld(values, elem), _ptr(index), _ld(index) if index is not None else 0, _ptr(meta),
        _ptr(status), _stream(stream)))
    return values, index, meta


def decompress(values: torch.Tensor, index: torch.Tensor, K: int, stream=None,
               elem: str | None = None) -> torch.Tensor:
    """The dense M x K operand (elem="s4" / "u4": M x K/2 packed bytes)."""
    t = _elem_code(values, elem)
    per = 2 if elem in PACKED4 else 1
    M = values.shape[0]
    A = torch.empty((M, K // per), dtype=values.dtype, device=values.device)
    _check("sp24_decompress", lib().sp24_decompress(
        t, M, K, _ptr(values), _ld(values, elem), _ptr(index), _ld(index), _ptr(A),
        _ld(A, elem), _stream(stream)))
    return A


def meta_bytes(dtype, M: int, K: int) -> int:
    return int(lib().sp24_meta_bytes(_code(dtype), M, K))


def meta_prepare(index: torch.Tensor, dtype, M: int, K: int, stream=None) -> torch.Tensor:
    nbytes = meta_bytes(dtype, M, K)
    meta = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=index.device)
    _check("sp24_meta_prepare", lib().sp24_meta_prepare(
        _code(dtype), M, K, _ptr(index), _ld(index), _ptr(meta), _stream(stream)))
    return meta


def workspace_bytes(a_dtype, b_dtype, M: int, N: int, K: int) -> int:
    """Device workspace sp24_mma needs (non-zero only for integer operands); the types
    are torch dtypes or names ("s4", "u4", ...)."""
    return int(lib().sp24_mma_workspace_bytes(_code(a_dtype), _code(b_dtype), M, N, K))


def mma(values: torch.Tensor, meta: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None,
        out_dtype=None, out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
        status: torch.Tensor | None = None, stream=None, a_elem: str | None = None,
        b_elem: str | None = None) -> torch.Tensor:
    """D = expand(values, meta) @ B + C  (values M x K/2, B K x N, C/D M x N).

    Float operands give f32 (default) or bf16 output; integer operands give int32.
    a_elem / b_elem = "s4" / "u4": that operand is packed 4-bit (values M x K/4 bytes,
    B K x N/2 bytes)."""
    return _mma("sp24_mma", values, (_ptr(meta),), B, C, out_dtype, out, workspace, status,
                stream, a_elem, b_elem)


def mma_index(values: torch.Tensor, index: torch.Tensor, B: torch.Tensor,
              C: torch.Tensor | None = None, out_dtype=None, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, status: torch.Tensor | None = None,
              stream=None, a_elem: str | None = None, b_elem: str | None = None) -> torch.Tensor:
    """mma() with the metadata read from the canonical index (M x K/32 int32, as compress()
    returns it) instead of the image; no meta_prepare pass."""
    return _mma("sp24_mma_index", values, (_ptr(index), _ld(index)), B, C, out_dtype, out,
                workspace, status, stream, a_elem, b_elem)


def _mma(fn, values, meta_args, B, C, out_dtype, out, workspace, status, stream, a_elem, b_elem):
    ta, tb = _elem_code(values, a_elem), _elem_code(B, b_elem)
    M = values.shape[0]
    K, N = B.shape[0], B.shape[1] * (2 if b_elem in PACKED4 else 1)
    integer = values.dtype in (torch.int8, torch.uint8)
    if out is None:
        if out_dtype is None:
            out_dtype = torch.int32 if integer else torch.float32
        out = torch.empty((M, N), dtype=out_dtype, device=B.device)
    tc = _code(C.dtype) if C is not None else _code(out.dtype if integer else torch.float32)
    ws_bytes = int(lib().sp24_mma_workspace_bytes(ta, tb, M, N, K))
    if ws_bytes and workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=B.device)
    _check(fn, getattr(lib(), fn)(
        ta, tb, tc, _code(out.dtype), M, N, K,
        _ptr(values), _ld(values, a_elem), *meta_args, _ptr(B), _ld(B, b_elem), _ptr(C),
        _ld(C) if C is not None else N, _ptr(out), _ld(out), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(),
        _ptr(status), _stream(stream)))
    return out


def mma_batched(values: torch.Tensor, meta: torch.Tensor, B: torch.Tensor,
                C: torch.Tensor | None = None, out_dtype=torch.float32,
                out: torch.Tensor | None = None, status: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """D[b] = expand(values[b], meta[b]) @ B[b] + C[b] for every b, in one launch.

    values: (batch, M, K/2), meta: (batch, sp24_meta_bytes) uint8, B: (batch, K, N),
    C / out: (batch, M, N); float operands only.  Rows of each matrix must be contiguous
    in their last dimension (the leading dimension is stride(1))."""
    batch, M = values.shape[0], values.shape[1]
    K, N = B.shape[1], B.shape[2]
    if out is None:
        out = torch.empty((batch, M, N), dtype=out_dtype, device=B.device)
    tc = _code(C.dtype) if C is not None else _code(torch.float32)
    _check("sp24_mma_strided_batched", lib().sp24_mma_strided_batched(
        _code(values.dtype), _code(B.dtype), tc, _code(out.dtype), batch, M, N, K,
        _ptr(values), values.stride(1), values.stride(0), _ptr(meta),
        meta.stride(0) * meta.element_size(), _ptr(B), B.stride(1), B.stride(0), _ptr(C),
        C.stride(1) if C is not None else N, C.stride(0) if C is not None else 0,
        _ptr(out), out.stride(1), out.stride(0), _ptr(status), _stream(stream)))
    return out


def mma_grouped(items, out_dtype=torch.float32, status: torch.Tensor | None = None,
                stream=None) -> list:
    """D_g = expand(values_g, meta_g) @ B_g + C_g for problems of different shapes in one
    launch (per 32 problems).  items: sequence of (values, meta, B, C or None); float
    operands of one type.  Returns the list of D_g (M_g x N_g, out_dtype)."""
    items = list(items)
    if not items:
        return []
    outs, keep = [], []
    arr = (Problem * len(items))()
    ta = tb = tc = None
    for i, (values, meta, B, C) in enumerate(items):
        M, (K, N) = values.shape[0], B.shape
        D = torch.empty((M, N), dtype=out_dtype, device=B.device)
        outs.append(D)
        keep.extend([values, meta, B, C, D])
        ta, tb = _code(values.dtype), _code(B.dtype)
        if C is not None:
            tc = _code(C.dtype)
        arr[i] = Problem(M, N, K, values.data_ptr(), _ld(values), meta.data_ptr(), B.data_ptr(),
                         _ld(B), 0 if C is None else C.data_ptr(), N if C is None else _ld(C),
                         D.data_ptr(), _ld(D))
    _check("sp24_mma_grouped", lib().sp24_mma_grouped(
        ta, tb, tc if tc is not None else _code(torch.float32), _code(out_dtype), arr, len(items),
        _ptr(status), _stream(stream)))
    return outs


def mma_i8_noalloc(values: torch.Tensor, meta: torch.Tensor, B: torch.Tensor,
                   C: torch.Tensor | None = None, out: torch.Tensor | None = None,
                   status: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The 8-bit integer product through sp24_mma_i8_noalloc: no workspace is passed, the
    library's fixed scratch array is used (for callers that cannot allocate; see the
    header).  Only the output tensor is allocated here, and only if `out` is None."""
    M = values.shape[0]
    K, N = B.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.int32, device=B.device)
    _check("sp24_mma_i8_noalloc", lib().sp24_mma_i8_noalloc(
        _code(values.dtype), _code(B.dtype), _code(torch.int32), _code(out.dtype), M, N, K,
        _ptr(values), _ld(values), _ptr(meta), _ptr(B), _ld(B), _ptr(C),
        _ld(C) if C is not None else N, _ptr(out), _ld(out), _ptr(status), _stream(stream)))
    return out


class SparseMatrix:
    """A compressed 2:4 operand: values + canonical index + the GEMM's metadata image."""

    def __init__(self, values, index, meta, K):
        self.values, self.index, self.meta, self.K = values, index, meta, K

    @property
    def shape(self):
        return (self.values.shape[0], self.K)

    @classmethod
    def from_dense(cls, A, mode="exact", mask=None, status=None, stream=None):
        values, index, meta = compress_meta(A, mode=mode, mask=mask, status=status,
                                            stream=stream)
        return cls(values, index, meta, A.shape[1])

    def to_dense(self, stream=None):
        return decompress(self.values, self.index, self.K, stream=stream)

    def matmul(self, B, C=None, out_dtype=None, status=None, stream=None):
        return mma(self.values, self.meta, B, C, out_dtype=out_dtype, status=status,
                   stream=stream)

    def state_dict(self) -> dict:
        """The compressed operand as plain tensors (for torch.save): the kept values, the
        canonical index, the metadata image and the dense K.  A compressed weight is kept and
        reloaded this way instead of being compressed again."""
        return {"values": self.values, "index": self.index, "meta": self.meta,
                "K": torch.tensor(self.K, dtype=torch.int64)}

    @classmethod
    def from_state_dict(cls, state: dict, device=None) -> "SparseMatrix":
        """Rebuild from state_dict() (the tensors moved to `device` if one is given)."""
        move = (lambda t: t.to(device)) if device is not None else (lambda t: t)
        return cls(move(state["values"]), move(state["index"]), move(state["meta"]),
                   int(state["K"]))
