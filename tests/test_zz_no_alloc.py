"""sp24_mma_i8_noalloc -- the integer product for callers that cannot allocate device
memory (its scratch is a fixed array inside the library) -- against the regular sp24_mma
with a workspace, through the C ABI, on two calls in a row with different data.  This file
is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import inputs
import structured_sparse_matrix_gb300 as sp

pytestmark = pytest.mark.gpu

S8, U8, S32 = 4, 5, 7


def _operands(ta, M, N, K, seed):
    c = inputs.case(ta, "s8", M, N, K, seed=seed, dist="full", tc="s32")
    A = c["A"].cuda()
    values, index = sp.compress(A, mode="mask", mask=c["mask"].cuda())
    meta = sp.meta_prepare(index, A.dtype, M, K)
    return values, meta, c["B"].cuda(), c["C"].cuda()


def _noalloc(ta, values, meta, B, C, D):
    M, N, K = values.shape[0], B.shape[1], B.shape[0]
    return sp.lib().sp24_mma_i8_noalloc(
        ta, S8, S32, S32, M, N, K, sp._ptr(values), values.stride(0), sp._ptr(meta),
        sp._ptr(B), B.stride(0), sp._ptr(C), C.stride(0), sp._ptr(D), D.stride(0), None,
        sp._stream())


def test_noalloc_matches_regular_entry_point_on_two_calls():
    # two calls in a row, different data and types: stale scratch contents must not matter
    for ta, ta_name, (M, N, K), seed in ((S8, "s8", (200, 144, 1056), 1),
                                         (U8, "u8", (130, 272, 2080), 2)):
        values, meta, B, C = _operands(ta_name, M, N, K, seed)
        ref = sp.mma(values, meta, B, C)                      # regular entry, workspace
        D = torch.full((M, N), 12345, dtype=torch.int32, device="cuda")
        assert _noalloc(ta, values, meta, B, C, D) == 0
        torch.cuda.synchronize()
        assert torch.equal(D, ref)                            # integer results: exact


def test_noalloc_rejects_problems_beyond_its_scratch():
    M = N = K = 4096  # needs 8 MiB + 32 MiB of widened operands, more than the array
    assert sp.lib().sp24_mma_workspace_bytes(S8, S8, M, N, K) > sp.lib().sp24_mma_workspace_bytes(S8, S8, 1, 1, 32)
    fake = ctypes.c_void_p(0x10000)
    rc = sp.lib().sp24_mma_i8_noalloc(S8, S8, S32, S32, M, N, K, fake, K // 2, fake, fake, N,
                                      None, N, fake, N, None, None)
    assert rc == 8  # SP24_ERR_SCRATCH_TOO_SMALL, nothing enqueued
    assert b"scratch" in sp.lib().sp24_status_string(rc)
