"""Shared helpers for the GPU-vs-oracle parity tests (CUDA path through the C ABI on one
side, the CPU oracle on the other, fed the same seeded inputs)."""
from __future__ import annotations

import numpy as np
import torch

import inputs
import oracle
import structured_sparse_matrix_gb300 as sp

REL, ABS = 1e-4, 1e-6  # float acceptance: |D - D_ref| <= REL * sum_k |a b| + ABS


def dev(t):
    return None if t is None else t.cuda()


def index_np(index_t: torch.Tensor) -> np.ndarray:
    return index_t.cpu().numpy().view(np.uint32)


def sample_rows(M: int) -> np.ndarray:
    """Rows 0..127, the last 128 and every 61st row: covers first/last tiles and a
    spread of interior tiles and lanes."""
    rows = set(range(min(128, M))) | set(range(max(0, M - 128), M)) | set(range(0, M, 61))
    return np.array(sorted(rows), dtype=np.int64)


def tile_quarter_rows(M: int) -> np.ndarray:
    """One row from each 32-row quarter of every 128-row tile (the four lane quarters of
    every CTA's accumulator), at a lane offset that varies from tile to tile."""
    rows = [t * 128 + q * 32 + (t * 7 + q * 13) % 32
            for t in range((M + 127) // 128) for q in range(4)]
    return np.array([r for r in rows if r < M], dtype=np.int64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -126)
    return np.exp2(e - 7)


def f16_ulp(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    e = np.maximum(e, -14)
    return np.exp2(e - 10)


OUT_KIND = {torch.float32: None, torch.bfloat16: "bf16", torch.float16: "f16"}


def check_float(D: np.ndarray, Dref: np.ndarray, S: np.ndarray, out, what: str):
    """Float parity: f32 output within REL*S + ABS; 16-bit output (out = "bf16" / "f16",
    or True for bf16) compared with the round-to-nearest-even value of the exact result,
    plus one ulp of that format (the f32 accumulation error may flip a rounding)."""
    D = np.asarray(D, dtype=np.float64)
    if out is True:
        out = "bf16"
    if out == "bf16":
        ref = oracle.decode("bf16", oracle.round_bf16(Dref))
        tol = REL * S + ABS + bf16_ulp(ref)
    elif out == "f16":
        ref = oracle.decode("f16", oracle.round_f16(Dref))
        tol = REL * S + ABS + f16_ulp(ref)
    else:
        ref = Dref
        tol = REL * S + ABS
    with np.errstate(invalid="ignore"):  # inf - inf where both overflowed
        err = np.abs(D - ref)
    bad = ~((err <= tol) | (D == ref))  # equal infinities (a 16-bit overflow) agree
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first at "
            f"{tuple(int(v) for v in i)}: got {D[tuple(i)]!r}, want {ref[tuple(i)]!r}, "
            f"tol {tol[tuple(i)]!r}")


def gpu_compress(c: dict, mode: str):
    A = dev(c["A"])
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = dev(c["mask"]) if mode == "mask" else None
    values, index = sp.compress(A, mode=mode, mask=mask, status=status)
    return values, index, status


def run_case(c: dict, mode: str = "mask", out_dtype=torch.float32, rows=None, check=True,
             fused: bool = False, by_index: bool = False):
    """Compress + meta_prepare + mma on the GPU (fused: compress_meta), oracle on the CPU,
    compare.  by_index: the product reads the canonical index (mma_index), and must equal
    the product on the image bit for bit."""
    ta, tb = c["ta"], c["tb"]
    M, N, K = c["M"], c["N"], c["K"]
    if fused:
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        values, index, meta = sp.compress_meta(
            dev(c["A"]), mode=mode, mask=dev(c["mask"]) if mode == "mask" else None,
            status=status)
    else:
        values, index, status = gpu_compress(c, mode)
        meta = sp.meta_prepare(index, c["A"].dtype, M, K)
    B = dev(c["B"])
    C = dev(c["C"])
    D = sp.mma(values, meta, B, C, out_dtype=out_dtype)
    if by_index:
        D_img = D
        D = sp.mma_index(values, index, B, C, out_dtype=out_dtype, status=status)
        torch.cuda.synchronize()
        assert torch.equal(D.view(torch.uint8), D_img.view(torch.uint8)), \
            "product on the canonical index differs from the product on the image"
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # oracle: its own compression of the same dense input, then its own product
    mask_np = c["mask"].numpy() if mode == "mask" else None
    v_ref, i_ref, _ = oracle.compress(inputs.bits(c["A"]), ta, mode, mask=mask_np)
    assert np.array_equal(index_np(index), i_ref), "index differs from the oracle"
    assert np.array_equal(inputs.bits(values.cpu()), v_ref), "values differ from the oracle"
    if rows is None:
        rows = np.arange(M)
    Dg = D.float().cpu().numpy()[rows] if out_dtype != torch.int32 else D.cpu().numpy()[rows]
    C_np = None if c["C"] is None else inputs.bits(c["C"])
    if ta in ("s8", "u8"):
        Dref = oracle.mma_i64(v_ref, i_ref, inputs.bits(c["B"]), C_np, ta, tb, K, rows=rows)
        if check:
            assert np.array_equal(Dg.astype(np.int64), oracle.wrap_i32(Dref).astype(np.int64))
        return Dg, Dref, None
    Dref, S = oracle.mma_f64(v_ref, i_ref, inputs.bits(c["B"]), C_np, ta, tb, K,
                             tc=c.get("tc") or "f32", rows=rows)
    if check:
        check_float(Dg, Dref, S, OUT_KIND[out_dtype], f"{ta} {M}x{N}x{K}")
    return Dg, Dref, S
