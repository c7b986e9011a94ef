"""Plain CPU oracle for the 2:4 structured-sparse multiply-accumulate D = A_sp * B + C.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import this package.  The CUDA
library never links, loads or calls it, and it shares no code with the CUDA library.

The arithmetic lives in ``sp24_oracle.c`` (plain C, double / int64, OpenMP over rows);
this module only builds that file with gcc on first use and marshals numpy arrays.
Citations for every function are in ``sp24_oracle.h``.

Arrays carry raw element bits: f16/bf16 as ``uint16``, e4m3/e5m2/u8 as ``uint8``, s8 as
``int8`` (or ``uint8``), C as ``float32`` / ``int32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sp24_oracle.c")
_HDR = os.path.join(_HERE, "sp24_oracle.h")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3, "s8": 4, "u8": 5, "f32": 6, "s32": 7,
          "s4": 8, "u4": 9}  # 4-bit: one element per byte, pattern in the low nibble
MODES = {"exact": 0, "mask": 1, "magnitude": 2}
ELEM_BYTES = {"f16": 2, "bf16": 2, "e4m3": 1, "e5m2": 1, "s8": 1, "u8": 1, "f32": 4, "s32": 4,
              "s4": 1, "u4": 1}
FLAG_NOT_2_4 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile sp24_oracle.c into _build/liboracle.so (gcc, -fopenmp)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    newest = max(os.path.getmtime(_SRC), os.path.getmtime(_HDR))
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= newest:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            i64, p, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
            L.or_decode.restype = ctypes.c_double
            L.or_decode.argtypes = [i32, ctypes.c_uint32]
            L.or_round_bf16.restype = ctypes.c_uint16
            L.or_round_bf16.argtypes = [ctypes.c_double]
            L.or_wrap_i32.restype = ctypes.c_int32
            L.or_wrap_i32.argtypes = [i64]
            L.or_compress.restype = i64
            L.or_compress.argtypes = [i32, i64, i64, p, i64, p, i64, i32, p, i64, p, i64, p]
            L.or_decompress.restype = None
            L.or_decompress.argtypes = [i32, i64, i64, p, i64, p, i64, p, i64]
            L.or_mma_f64.restype = i32
            L.or_mma_f64.argtypes = [i32, i32, i64, i64, i64, p, i64, p, i64, p, i64,
                                     i32, p, i64, p, i64, p, p]
            L.or_mma_i64.restype = i32
            L.or_mma_i64.argtypes = [i32, i32, i64, i64, i64, p, i64, p, i64, p, i64,
                                     p, i64, p, i64, p]
            L.or_decode_array.restype = None
            L.or_decode_array.argtypes = [i32, p, i64, p]
            L.or_round_bf16_array.restype = None
            L.or_round_bf16_array.argtypes = [p, i64, p]
            L.or_round_f16_array.restype = None
            L.or_round_f16_array.argtypes = [p, i64, p]
            L.or_wrap_i32_array.restype = None
            L.or_wrap_i32_array.argtypes = [p, i64, p]
            L.or_num_threads.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a):
    return None if a is None else np.ascontiguousarray(a)


def num_threads() -> int:
    return int(lib().or_num_threads())


_BITS_DTYPE = {1: np.uint8, 2: np.uint16, 4: np.uint32}


def decode(dtype: str, bits) -> np.ndarray:
    """Exact float64 value of each stored element (bits: any integer array)."""
    nb = ELEM_BYTES[dtype]
    arr = np.asarray(bits)
    flat = np.ascontiguousarray(
        (arr.astype(np.int64).ravel() & ((1 << (8 * nb)) - 1)).astype(_BITS_DTYPE[nb]))
    out = np.empty(flat.size, dtype=np.float64)
    lib().or_decode_array(DTYPES[dtype], _ptr(flat), flat.size, _ptr(out))
    return out.reshape(arr.shape)


def round_bf16(x) -> np.ndarray:
    """bfloat16 bit patterns of x rounded to nearest, ties to even."""
    arr = np.asarray(x, dtype=np.float64)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.uint16)
    lib().or_round_bf16_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(arr.shape)


def round_f16(x) -> np.ndarray:
    """IEEE binary16 bit patterns of x rounded to nearest, ties to even."""
    arr = np.asarray(x, dtype=np.float64)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.uint16)
    lib().or_round_f16_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(arr.shape)


def wrap_i32(x) -> np.ndarray:
    """Two's-complement 32-bit wrap of exact integer results."""
    arr = np.asarray(x, dtype=np.int64)
    flat = np.ascontiguousarray(arr.ravel())
    out = np.empty(flat.size, dtype=np.int32)
    lib().or_wrap_i32_array(_ptr(flat), flat.size, _ptr(out))
    return out.reshape(arr.shape)


def compress(A: np.ndarray, dtype: str, mode: str = "exact", mask: np.ndarray | None = None):
    """Dense M x K bits -> (values M x K/2, index M x ceil(K/32) uint32, flags M x K/4)."""
    A = _c(A)
    M, K = A.shape
    if K % 4:
        raise ValueError("K must be a multiple of 4")
    if A.dtype.itemsize != ELEM_BYTES[dtype]:
        raise ValueError(f"{dtype} wants {ELEM_BYTES[dtype]}-byte elements")
    values = np.zeros((M, K // 2), dtype=A.dtype)
    words = (K // 4 + 7) // 8
    index = np.zeros((M, words), dtype=np.uint32)
    flags = np.zeros((M, K // 4), dtype=np.uint8)
    m = None
    if mode == "mask":
        if mask is None:
            raise ValueError("mask mode needs a mask")
        m = _c(np.asarray(mask).astype(np.uint8))
    n = lib().or_compress(DTYPES[dtype], M, K, _ptr(A), K, _ptr(m), K, MODES[mode],
                          _ptr(values), K // 2, _ptr(index), words, _ptr(flags))
    if n < 0:
        raise ValueError("or_compress rejected its arguments")
    return values, index, flags


def decompress(values: np.ndarray, index: np.ndarray, dtype: str, K: int) -> np.ndarray:
    values = _c(values)
    index = _c(np.asarray(index, dtype=np.uint32))
    M = values.shape[0]
    A = np.zeros((M, K), dtype=values.dtype)
    lib().or_decompress(DTYPES[dtype], M, K, _ptr(values), values.shape[1], _ptr(index),
                        index.shape[1], _ptr(A), K)
    return A


def _rows_arg(rows, M):
    if rows is None:
        return None, M
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    if r.size and (r.min() < 0 or r.max() >= M):
        raise ValueError("row index out of range")
    return r, int(r.size)


def mma_f64(values, index, B, C, ta: str, tb: str, K: int, tc: str = "f32", rows=None):
    """(D, S): D = expand(values, index) @ B + C in float64, S = sum_k |a_ik b_kj|."""
    values, B = _c(values), _c(B)
    index = _c(np.asarray(index, dtype=np.uint32))
    C = _c(C)
    M = values.shape[0]
    N = B.shape[1]
    r, nr = _rows_arg(rows, M)
    D = np.zeros((nr, N), dtype=np.float64)
    S = np.zeros((nr, N), dtype=np.float64)
    rc = lib().or_mma_f64(DTYPES[ta], DTYPES[tb], M, N, K, _ptr(values), values.shape[1],
                          _ptr(index), index.shape[1], _ptr(B), B.shape[1], DTYPES[tc],
                          _ptr(C), 0 if C is None else C.shape[1], _ptr(r), nr,
                          _ptr(D), _ptr(S))
    if rc != 0:
        raise ValueError(f"or_mma_f64 failed ({rc})")
    return D, S


def mma_i64(values, index, B, C, ta: str, tb: str, K: int, rows=None) -> np.ndarray:
    """Exact int64 D = expand(values, index) @ B + C for s8/u8/s4/u4 operands."""
    values, B = _c(values), _c(B)
    index = _c(np.asarray(index, dtype=np.uint32))
    C = _c(C)
    M = values.shape[0]
    N = B.shape[1]
    r, nr = _rows_arg(rows, M)
    D = np.zeros((nr, N), dtype=np.int64)
    rc = lib().or_mma_i64(DTYPES[ta], DTYPES[tb], M, N, K, _ptr(values), values.shape[1],
                          _ptr(index), index.shape[1], _ptr(B), B.shape[1], _ptr(C),
                          0 if C is None else C.shape[1], _ptr(r), nr, _ptr(D))
    if rc != 0:
        raise ValueError(f"or_mma_i64 failed ({rc})")
    return D


def tolerance_ok(D, D_ref, S, rel: float = 1e-4, abs_: float = 1e-6):
    """Elementwise |D - D_ref| <= rel * S + abs_ (the float-path acceptance bound)."""
    D = np.asarray(D, dtype=np.float64)
    return np.abs(D - D_ref) <= rel * S + abs_
