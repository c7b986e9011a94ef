"""GPU compression, decompression and metadata re-layout against the oracle (bit-exact)."""
import numpy as np
import pytest
import torch

import inputs
import oracle
import structured_sparse_matrix_gb300 as sp
from parity import dev, gpu_compress, index_np

pytestmark = pytest.mark.gpu

TYPES = ["f16", "bf16", "e4m3", "e5m2", "s8", "u8"]


def _dense_case(ta, M, K, seed, with_zeros):
    """Random dense A (no mask applied) -- exercises every mode's selection rules."""
    dist = "full" if ta in ("s8", "u8") else ("int4" if with_zeros else "normal")
    if ta in ("e4m3", "e5m2") and with_zeros:
        dist = "normal"
    A = inputs.values((M, K), ta, dist, inputs.gen(seed))
    m = inputs.keep_mask(M, K, inputs.gen(seed + 1))
    return {"A": A, "mask": m, "ta": ta, "M": M, "K": K}


@pytest.mark.parametrize("ta", TYPES)
@pytest.mark.parametrize("mode", ["exact", "mask", "magnitude"])
def test_compress_matches_oracle(ta, mode):
    # 37 rows and K = 160 (5 index words): ragged against every block and warp size
    c = _dense_case(ta, 37, 160, seed=21, with_zeros=True)
    if mode == "exact":
        # a 2:4 input (what exact mode is for) with some kept values zero
        c["A"] = inputs.apply_mask(c["A"], c["mask"])
    values, index, status = gpu_compress(c, mode)
    torch.cuda.synchronize()
    v_ref, i_ref, flags = oracle.compress(inputs.bits(c["A"]), ta, mode,
                                          mask=c["mask"].numpy() if mode == "mask" else None)
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.bits(values.cpu()), v_ref)
    assert bool(status.item() & sp.DEV_NOT_2_4) == bool(flags.any())


@pytest.mark.parametrize("ta", ["bf16", "e4m3", "s8"])
def test_exact_mode_flags_dense_input(ta):
    # a fully dense input has groups with > 2 non-zeros: flagged, two lowest kept
    c = _dense_case(ta, 16, 64, seed=5, with_zeros=False)
    values, index, status = gpu_compress(c, "exact")
    torch.cuda.synchronize()
    v_ref, i_ref, flags = oracle.compress(inputs.bits(c["A"]), ta, "exact")
    assert flags.any()
    assert status.item() & sp.DEV_NOT_2_4
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.bits(values.cpu()), v_ref)


def test_exact_mode_fill_rules_f16():
    h = lambda v: int(np.float16(v).view(np.uint16))
    row = [0, 0, 0, 0, 0, 0, 0, h(5), 0, h(-2), 0, 0, h(1), h(2), h(3), 0,
           0x8000, h(7), 0, 0x8000, h(1), 0, 0, h(2), 0, 0, h(4), h(6), 0, h(1), h(1), 0]
    A = torch.tensor(np.array([row] * 3, dtype=np.uint16).view(np.int16)).view(torch.float16)
    c = {"A": A, "mask": None, "ta": "f16", "M": 3, "K": 32}
    values, index, status = gpu_compress(c, "exact")
    torch.cuda.synchronize()
    v_ref, i_ref, flags = oracle.compress(inputs.bits(A), "f16", "exact")
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.bits(values.cpu()), v_ref)
    assert status.item() & sp.DEV_NOT_2_4


def test_compress_fixed_pattern_index_literal():
    c = inputs.fixed_pattern_case()
    values, index, status = gpu_compress(c, "mask")
    torch.cuda.synchronize()
    assert status.item() == 0
    assert np.all(index_np(index) == 0x88888888)


def test_compress_padded_leading_dimensions():
    M, K = 40, 96
    big = inputs.values((M, K + 64), "bf16", "normal", inputs.gen(3)).cuda()
    A = big[:, 16:16 + K]                      # lda = K + 64, offset 32 bytes
    m = inputs.keep_mask(M, K, inputs.gen(4))
    Am = torch.where(m.cuda(), A, torch.zeros((), dtype=A.dtype, device="cuda"))
    big2 = torch.zeros((M, K + 64), dtype=torch.bfloat16, device="cuda")
    big2[:, 16:16 + K] = Am
    A2 = big2[:, 16:16 + K]
    values, index = sp.compress(A2, mode="exact")
    torch.cuda.synchronize()
    v_ref, i_ref, _ = oracle.compress(inputs.bits(Am.cpu()), "bf16", "exact")
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.bits(values.cpu()), v_ref)


@pytest.mark.parametrize("ta", TYPES)
def test_decompress_round_trip(ta):
    c = inputs.case(ta, ta, 50, 8, 192, seed=6, dist="full" if ta in ("s8", "u8") else "normal")
    values, index, _ = gpu_compress(c, "mask")
    A = sp.decompress(values, index, 192)
    torch.cuda.synchronize()
    ref = oracle.decompress(inputs.bits(values.cpu()), index_np(index), ta, 192)
    assert np.array_equal(inputs.bits(A.cpu()), ref)
    assert np.array_equal(ref, inputs.bits(c["A"]))


def test_compress_full_size_bf16_4096_mask_mode():
    c = inputs.bf16_square()
    values, index, status = gpu_compress(c, "mask")
    torch.cuda.synchronize()
    assert status.item() == 0
    v_ref, i_ref, _ = oracle.compress(inputs.bits(c["A"]), "bf16", "mask", mask=c["mask"].numpy())
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.bits(values.cpu()), v_ref)


def test_prune_full_size_llm_weight():
    c = inputs.llm_layer(N=16)
    values, index, status = gpu_compress(c, "magnitude")
    torch.cuda.synchronize()
    v_ref, i_ref, _ = oracle.compress(inputs.bits(c["A"]), "bf16", "magnitude")
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(inputs.bits(values.cpu()), v_ref)


def test_empty_inputs_are_no_ops():
    A = torch.empty((0, 64), dtype=torch.float16, device="cuda")
    values, index = sp.compress(A)
    assert values.shape == (0, 32) and index.shape == (0, 2)


# --- metadata image: checked against an independent restatement of the documented layout

def _meta_image_np(index: np.ndarray, M: int, K: int, eight_bit: bool) -> np.ndarray:
    """Image layout: per (128-row tile, stage) one [128 lanes][W words] block holding each
    lane's words for the stage's 4 MMAs in MMA order (16-bit: one interleaved word per MMA,
    W = 4; FP8: the MMA's two canonical words, so a lane holds its row's 8 words of the
    stage, W = 8); the tiles cover M rounded up to 256 rows, padding is 0x44444444."""
    stage = 256 if eight_bit else 128
    mt, ks = 2 * -(-M // 256), -(-K // stage)
    canon = np.full((mt * 128, ks * stage // 32), 0x44444444, dtype=np.uint64)
    canon[:M, :K // 32] = index[:, :K // 32]
    out = []
    for t in range(mt):
        for s in range(ks):
            if eight_bit:
                blk = canon[t * 128:(t + 1) * 128, s * 8:s * 8 + 8]
            else:
                blk = np.zeros((128, 4), dtype=np.uint64)
                for j in range(4):
                    w = s * 4 + j
                    for lane in range(128):
                        band, l = divmod(lane, 16)
                        rA = t * 128 + band * 16 + (l % 8)
                        h = l // 8
                        lo = (int(canon[rA, w]) >> (16 * h)) & 0xFFFF
                        hi = (int(canon[rA + 8, w]) >> (16 * h)) & 0xFFFF
                        blk[lane, j] = lo | (hi << 16)
            out.append(np.asarray(blk).reshape(-1))
    return np.concatenate(out).astype(np.uint32)


@pytest.mark.parametrize("ta,M,K", [("bf16", 200, 352), ("e4m3", 130, 544), ("f16", 64, 128)])
def test_meta_prepare_layout(ta, M, K):
    c = inputs.case(ta, ta, M, 8, K, seed=9)
    values, index, _ = gpu_compress(c, "mask")
    meta = sp.meta_prepare(index, c["A"].dtype, M, K)
    torch.cuda.synchronize()
    got = meta.cpu().numpy().view(np.uint32)
    want = _meta_image_np(index_np(index), M, K, ta in ("e4m3", "e5m2", "s8", "u8"))
    assert got.shape == want.shape
    assert np.array_equal(got, want)


# --- compression and the metadata image in one pass (sp24_compress_meta) -------------------

def _fused_inputs(ta, M, K, seed, mode):
    """Dense operand for ta (4-bit types as one nibble per byte), its mask, and the tensor
    handed to the library (4-bit types packed two per byte)."""
    mask = inputs.keep_mask(M, K, inputs.gen(seed + 1))
    if ta in ("s4", "u4"):
        dense = inputs.gen_nibbles((M, K), inputs.gen(seed))
        if mode == "exact":
            dense = np.where(mask.numpy(), dense, 0).astype(np.uint8)
        return dense, mask, torch.from_numpy(inputs.pack4(dense)).cuda()
    c = _dense_case(ta, M, K, seed, with_zeros=True)
    A = inputs.apply_mask(c["A"], mask) if mode == "exact" else c["A"]
    return inputs.bits(A), mask, A.cuda()


@pytest.mark.parametrize("ta", TYPES + ["s4", "u4"])
@pytest.mark.parametrize("mode", ["exact", "mask", "magnitude"])
@pytest.mark.parametrize("M,K", [(37, 160), (200, 352), (257, 544)])
def test_compress_meta_matches_oracle(ta, mode, M, K):
    # ragged against the band (16 rows), the tile pair (256 rows) and the stage (128 / 256 K)
    dense, mask, A = _fused_inputs(ta, M, K, seed=M + K, mode=mode)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    elem = ta if ta in ("s4", "u4") else None
    values, index, meta = sp.compress_meta(A, mode=mode,
                                           mask=mask.cuda() if mode == "mask" else None,
                                           status=status, elem=elem)
    torch.cuda.synchronize()
    v_ref, i_ref, flags = oracle.compress(dense, ta, mode,
                                          mask=mask.numpy() if mode == "mask" else None)
    got_v = values.cpu().numpy() if elem else inputs.bits(values.cpu())
    if elem:
        got_v = inputs.unpack4(got_v)
    assert np.array_equal(index_np(index), i_ref)
    assert np.array_equal(got_v, v_ref)
    assert bool(status.item() & sp.DEV_NOT_2_4) == bool(flags.any())
    want = _meta_image_np(i_ref, M, K, ta in ("e4m3", "e5m2"))
    got = meta.cpu().numpy().view(np.uint32)
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_compress_meta_without_index_and_padded_pitch():
    M, K = 130, 256
    big = inputs.values((M, K + 64), "bf16", "normal", inputs.gen(31)).cuda()
    A = big[:, 32:32 + K]
    values, index, meta = sp.compress_meta(A, mode="magnitude", with_index=False)
    v2, i2 = sp.compress(A, mode="magnitude")
    m2 = sp.meta_prepare(i2, torch.bfloat16, M, K)
    torch.cuda.synchronize()
    assert index is None
    assert torch.equal(values, v2) and torch.equal(meta, m2)


def test_compress_meta_full_size_llm_weight():
    # the LLM layer's weight (14336 x 4096): image equal to the separate re-layout's
    c = inputs.llm_layer(N=16)
    A = c["A"].cuda()
    values, index, meta = sp.compress_meta(A, mode="magnitude")
    v2, i2 = sp.compress(A, mode="magnitude")
    m2 = sp.meta_prepare(i2, torch.bfloat16, A.shape[0], A.shape[1])
    torch.cuda.synchronize()
    assert torch.equal(index, i2) and torch.equal(values, v2) and torch.equal(meta, m2)
    v_ref, i_ref, _ = oracle.compress(inputs.bits(c["A"]), "bf16", "magnitude")
    assert np.array_equal(index_np(index), i_ref)
