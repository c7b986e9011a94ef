"""4-bit integer operands (s4, u4; two elements per byte, element 2i in the low nibble):
compression, decompression, the metadata image and the exact sparse product against the
oracle, which holds one 4-bit element per byte ("RDNA4 sparse WMMA builtins", "INT4 and
UINT4 inputs")."""
import numpy as np
import pytest
import torch

import inputs
import oracle
import structured_sparse_matrix_gb300 as sp
from parity import index_np, sample_rows

pytestmark = pytest.mark.gpu

T4 = ["s4", "u4"]


def _packed(nib: np.ndarray, pitch_bytes: int | None = None) -> torch.Tensor:
    """One-nibble-per-byte array -> packed uint8 tensor on the GPU (optionally a view of a
    wider buffer, so that the row pitch exceeds the row)."""
    p = inputs.pack4(nib)
    if pitch_bytes is None:
        return torch.from_numpy(np.ascontiguousarray(p)).cuda()
    buf = np.full((p.shape[0], pitch_bytes), 0xA5, dtype=np.uint8)  # junk in the pad
    buf[:, :p.shape[1]] = p
    return torch.from_numpy(buf).cuda()[:, :p.shape[1]]


def _mask_nibbles(nib: np.ndarray, mask: torch.Tensor) -> np.ndarray:
    return np.where(mask.numpy(), nib, 0).astype(np.uint8)


@pytest.mark.parametrize("ta", T4)
@pytest.mark.parametrize("mode", ["exact", "mask", "magnitude"])
def test_compress4_matches_oracle(ta, mode):
    # 37 rows, K = 160: five chunks of 32 elements a row, ragged against block and warp
    M, K = 37, 160
    nib = inputs.gen_nibbles((M, K), inputs.gen(41))
    mask = inputs.keep_mask(M, K, inputs.gen(42))
    if mode == "exact":
        nib = _mask_nibbles(nib, mask)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    values, index = sp.compress(_packed(nib), mode=mode,
                                mask=mask.cuda() if mode == "mask" else None, status=status,
                                elem=ta)
    torch.cuda.synchronize()
    v_ref, i_ref, flags = oracle.compress(nib, ta, mode,
                                          mask=mask.numpy() if mode == "mask" else None)
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.unpack4(values.cpu().numpy()), v_ref)
    assert bool(status.item() & sp.DEV_NOT_2_4) == bool(flags.any())


@pytest.mark.parametrize("ta", T4)
def test_compress4_exact_flags_dense_and_magnitude_extremes(ta):
    # every nibble pattern in every position: dense groups are flagged in exact mode; in
    # magnitude mode s4's -8 is the largest |x|
    M, K = 16, 64
    nib = (np.arange(M * K, dtype=np.int64).reshape(M, K) * 7 % 16).astype(np.uint8)
    nib[0, :4] = [8, 7, 0, 9]        # s4: -8, 7, 0, -7
    nib[1, :4] = [15, 1, 8, 15]      # s4: -1, 1, -8, -1
    for mode in ("exact", "magnitude"):
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        values, index = sp.compress(_packed(nib), mode=mode, status=status, elem=ta)
        torch.cuda.synchronize()
        v_ref, i_ref, flags = oracle.compress(nib, ta, mode)
        assert np.array_equal(index_np(index), i_ref), mode
        assert np.array_equal(inputs.unpack4(values.cpu().numpy()), v_ref), mode
        assert bool(status.item() & sp.DEV_NOT_2_4) == bool(flags.any()), mode
        if mode == "exact":
            assert flags.any()


@pytest.mark.parametrize("ta", T4)
def test_decompress4_round_trip(ta):
    M, K = 50, 192
    mask = inputs.keep_mask(M, K, inputs.gen(8))
    nib = _mask_nibbles(inputs.gen_nibbles((M, K), inputs.gen(7)), mask)
    values, index = sp.compress(_packed(nib), mode="mask", mask=mask.cuda(), elem=ta)
    A = sp.decompress(values, index, K, elem=ta)
    torch.cuda.synchronize()
    got = inputs.unpack4(A.cpu().numpy())
    ref = oracle.decompress(inputs.unpack4(values.cpu().numpy()), index_np(index), ta, K)
    assert np.array_equal(got, ref)
    assert np.array_equal(ref, nib)


def test_compress4_padded_pitch_and_short_rows():
    # K = 32: values rows are 8 bytes (the binding pads their pitch); A read from a view
    # whose pitch is 48 bytes with junk in the pad
    M, K = 9, 32
    mask = inputs.keep_mask(M, K, inputs.gen(12))
    nib = _mask_nibbles(inputs.gen_nibbles((M, K), inputs.gen(11)), mask)
    values, index = sp.compress(_packed(nib, pitch_bytes=48), mode="exact", elem="s4")
    torch.cuda.synchronize()
    v_ref, i_ref, _ = oracle.compress(nib, "s4", "exact")
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.unpack4(values.cpu().numpy()), v_ref)


def test_meta4_uses_the_16_bit_layout():
    M, K = 130, 352
    mask = inputs.keep_mask(M, K, inputs.gen(14))
    nib = _mask_nibbles(inputs.gen_nibbles((M, K), inputs.gen(13)), mask)
    values, index = sp.compress(_packed(nib), mode="mask", mask=mask.cuda(), elem="u4")
    m4 = sp.meta_prepare(index, "u4", M, K)
    m16 = sp.meta_prepare(index, torch.bfloat16, M, K)
    torch.cuda.synchronize()
    assert m4.numel() == sp.meta_bytes(torch.bfloat16, M, K)
    assert torch.equal(m4, m16)


def _run4(ta, tb, M, N, K, seed, *, nib_a=None, nib_b=None, C=None, b_pitch=None, rows=None,
          by_index=False):
    mask = inputs.keep_mask(M, K, inputs.gen(seed + 1))
    if nib_a is None:
        nib_a = inputs.gen_nibbles((M, K), inputs.gen(seed))
    nib_a = _mask_nibbles(nib_a, mask)
    if nib_b is None:
        nib_b = inputs.gen_nibbles((K, N), inputs.gen(seed + 2))
    if C is None:
        C = torch.randint(-(1 << 20), 1 << 20, (M, N), generator=inputs.gen(seed + 3),
                          dtype=torch.int32)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    values, index = sp.compress(_packed(nib_a), mode="mask", mask=mask.cuda(), status=status,
                                elem=ta)
    meta = sp.meta_prepare(index, ta, M, K)
    D = sp.mma(values, meta, _packed(nib_b, b_pitch), C.cuda(), a_elem=ta, b_elem=tb)
    if by_index:  # the product on the canonical index must equal the one on the image
        D_idx = sp.mma_index(values, index, _packed(nib_b, b_pitch), C.cuda(), a_elem=ta,
                             b_elem=tb)
        torch.cuda.synchronize()
        assert torch.equal(D_idx, D)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    v_ref, i_ref, _ = oracle.compress(nib_a, ta, "mask", mask=mask.numpy())
    assert np.array_equal(index_np(index), i_ref)
    Dref = oracle.wrap_i32(oracle.mma_i64(v_ref, i_ref, nib_b, C.numpy(), ta, tb, K, rows=rows))
    Dg = D.cpu().numpy()
    if rows is not None:
        Dg = Dg[rows]
    assert np.array_equal(Dg, Dref)
    return Dg, Dref


@pytest.mark.parametrize("ta", T4)
@pytest.mark.parametrize("tb", T4)
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 96, 1056), (33, 64, 2080),
                                   (257, 288, 320)])
def test_mma4_exact(ta, tb, M, N, K):
    _run4(ta, tb, M, N, K, seed=M + N + K)


@pytest.mark.parametrize("ta,tb,M,N,K", [("s4", "u4", 200, 96, 1056), ("u4", "s4", 33, 288, 8320)])
def test_mma4_reads_the_canonical_index(ta, tb, M, N, K):
    # ragged M and K; the second case spans two 8192-K exact chunks
    _run4(ta, tb, M, N, K, seed=M + K, by_index=True)


def test_mma4_ragged_n_through_a_padded_b():
    # N = 100 (50 bytes a row) read from a 64-byte pitch with junk in the pad
    _run4("s4", "u4", 144, 100, 384, seed=3, b_pitch=64)


@pytest.mark.parametrize("ta,tb,a,b", [("s4", "s4", 8, 8), ("u4", "u4", 15, 15),
                                       ("u4", "s4", 15, 8), ("s4", "u4", 8, 15)])
def test_mma4_extreme_values_many_chunks(ta, tb, a, b):
    # every kept a and every b at an extreme (s4 -8 = nibble 8); K = 4096 spans four
    # 1024-K chunks of the integer accumulation
    M, N, K = 128, 160, 4096
    Dg, Dref = _run4(ta, tb, M, N, K, seed=9, nib_a=np.full((M, K), a, dtype=np.uint8),
                     nib_b=np.full((K, N), b, dtype=np.uint8),
                     C=torch.zeros((M, N), dtype=torch.int32))
    va = a - 16 if (ta == "s4" and a >= 8) else a
    vb = b - 16 if (tb == "s4" and b >= 8) else b
    assert np.all(Dref == (K // 2) * va * vb)


def test_mma4_large_sampled_rows():
    # a multi-wave shape (8192 x 4096 x 4096), checked on sampled rows
    M, N, K = 8192, 4096, 4096
    _run4("s4", "s4", M, N, K, seed=21, rows=sample_rows(M)[::4])
