"""sp24_mma_i8_noalloc -- the integer product for callers that cannot allocate device
memory at the call (its scratch is a fixed array inside the library) -- through the C ABI:
against the oracle directly, and against the regular sp24_mma (which takes a workspace)
on two calls in a row with different data, plus the size limit on both sides of it.
This file is collected last on purpose."""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import inputs
import oracle
import structured_sparse_matrix_gb300 as sp
from parity import index_np, sample_rows

pytestmark = pytest.mark.gpu

S8, U8, S32 = 4, 5, 7
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _scratch_limit() -> int:
    """SP24_NOALLOC_SCRATCH_BYTES as the public header defines it."""
    with open(os.path.join(ROOT, "include", "sp24.h")) as f:
        m = re.search(r"#define SP24_NOALLOC_SCRATCH_BYTES \((\d+)u \* 1024u \* 1024u\)", f.read())
    return int(m.group(1)) * 2**20


def _operands(ta, M, N, K, seed):
    c = inputs.case(ta, "s8", M, N, K, seed=seed, dist="full", tc="s32")
    A = c["A"].cuda()
    values, index = sp.compress(A, mode="mask", mask=c["mask"].cuda())
    meta = sp.meta_prepare(index, A.dtype, M, K)
    return c, values, index, meta, c["B"].cuda(), c["C"].cuda()


def _noalloc(ta, values, meta, B, C, D):
    M, N, K = values.shape[0], B.shape[1], B.shape[0]
    return sp.lib().sp24_mma_i8_noalloc(
        ta, S8, S32, S32, M, N, K, sp._ptr(values), values.stride(0), sp._ptr(meta),
        sp._ptr(B), B.stride(0), sp._ptr(C), C.stride(0), sp._ptr(D), D.stride(0), None,
        sp._stream())


def _oracle_rows(c, values, index, ta_name, rows):
    v = inputs.bits(values.cpu())
    i = index_np(index)
    ref = oracle.mma_i64(v, i, inputs.bits(c["B"]), inputs.bits(c["C"]), ta_name, "s8", c["K"],
                         rows=rows)
    return oracle.wrap_i32(ref).astype(np.int64)


def test_noalloc_matches_oracle_and_regular_entry_point_on_two_calls():
    # two calls in a row, different data and types: stale scratch contents must not matter
    for ta, ta_name, (M, N, K), seed in ((S8, "s8", (200, 144, 1056), 1),
                                         (U8, "u8", (130, 272, 2080), 2)):
        c, values, index, meta, B, C = _operands(ta_name, M, N, K, seed)
        ref = sp.mma(values, meta, B, C)                      # regular entry, workspace
        D = torch.full((M, N), 12345, dtype=torch.int32, device="cuda")
        assert _noalloc(ta, values, meta, B, C, D) == 0
        torch.cuda.synchronize()
        assert torch.equal(D, ref)                            # integer results: exact
        # and the oracle itself, on every row (exact, two's-complement wrap)
        want = _oracle_rows(c, values, index, ta_name, np.arange(M))
        assert np.array_equal(D.cpu().numpy().astype(np.int64), want)


def test_noalloc_just_under_its_scratch_limit():
    # 2048^3 s8: widened A 4 MiB + widened B 8 MiB = 12 MiB, inside the array
    M = N = K = 2048
    need = sp.lib().sp24_mma_workspace_bytes(S8, S8, M, N, K)
    assert 12 * 2**20 <= need <= _scratch_limit()
    c, values, index, meta, B, C = _operands("s8", M, N, K, 3)
    ref = sp.mma(values, meta, B, C)
    D = torch.full((M, N), -7, dtype=torch.int32, device="cuda")
    assert _noalloc(S8, values, meta, B, C, D) == 0
    torch.cuda.synchronize()
    assert torch.equal(D, ref)
    rows = sample_rows(M)
    assert np.array_equal(D.cpu().numpy()[rows].astype(np.int64),
                          _oracle_rows(c, values, index, "s8", rows))


def test_noalloc_rejects_problems_beyond_its_scratch():
    M = N = K = 4096  # widened A 16 MiB + widened B 32 MiB, more than the array
    assert sp.lib().sp24_mma_workspace_bytes(S8, S8, M, N, K) > _scratch_limit()
    assert _scratch_limit() == 16 * 2**20
    fake = ctypes.c_void_p(0x10000)
    rc = sp.lib().sp24_mma_i8_noalloc(S8, S8, S32, S32, M, N, K, fake, K // 2, fake, fake, N,
                                      None, N, fake, N, None, None)
    assert rc == 8  # SP24_ERR_SCRATCH_TOO_SMALL, nothing enqueued
    assert b"scratch" in sp.lib().sp24_status_string(rc)
