"""Seeded synthetic inputs for the 2:4 sparse multiply-accumulate.

This module only draws numbers: dense operands, 2:4 keep-masks, the C operand.  It holds
none of the method's arithmetic (no compression, no index packing, no product) and is
imported by both the tests / bench (to feed the CUDA library) and the oracle checks, so
the two sides see bit-identical inputs.

Workloads (all synthetic; the pages measure nothing on a public suite):
  fixed_pattern_case  f16 64x128 A with the fixed pattern that keeps positions 0 and 2 of
      each group, B 128x64 f16, C 64x64 f32, integers uniform in [-4, 4], one generator
      seeded 0 drawing A, B, C in that order (the pages' example kernel);
  bf16_square  bf16 M=N=K=4096, mask uniform over the six two-of-four patterns,
      A, B ~ N(0,1), C f32 ~ N(0,1);
  fp8_square  8192^3 FP8 (E4M3 x E4M3, E5M2 x E5M2), N(0,1) scaled per tensor to the
      format's maximum and rounded to nearest-even with saturation, random mask, no C;
  int8_square  8192^3 int8 (s8 x s8, u8 x s8), uniform over the full 8-bit range, random
      mask, C s32 uniform in [-2^20, 2^20];
  llm_layer  W bf16 14336x4096 ~ N(0, 0.02) (pruned by magnitude on the device),
      X bf16 4096xN ~ N(0,1), N in {16, 128, 2048}.
Seeds of the square cases and the layer: A=0, B=1, C=2, mask=3 (plus the size in the
generic helper).
"""
from __future__ import annotations

import numpy as np
import torch

# the six ways to keep two of four positions, in lexicographic order
PATTERNS = ((0, 1), (0, 2), (0, 3), (1, 2), (1, 3), (2, 3))

TORCH_DTYPE = {
    "f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn,
    "e5m2": torch.float8_e5m2, "s8": torch.int8, "u8": torch.uint8,
    "f32": torch.float32, "s32": torch.int32,
}
FMT_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed))
    return g


def keep_mask(M: int, K: int, g: torch.Generator | None, fixed: tuple | None = None) -> torch.Tensor:
    """Bool M x K keep-mask with exactly two True per group of four along K.

    fixed=(p0, p1) keeps the same two positions in every group; otherwise each group's
    pattern is drawn uniformly from PATTERNS."""
    assert K % 4 == 0
    G = K // 4
    table = torch.zeros(len(PATTERNS), 4, dtype=torch.bool)
    for n, (a, b) in enumerate(PATTERNS):
        table[n, a] = True
        table[n, b] = True
    if fixed is not None:
        pid = torch.full((M, G), PATTERNS.index(tuple(fixed)), dtype=torch.long)
    else:
        pid = torch.randint(0, len(PATTERNS), (M, G), generator=g)
    return table[pid].reshape(M, K)


def values(shape, dtype: str, dist: str, g: torch.Generator, std: float = 1.0) -> torch.Tensor:
    """Dense tensor of `dtype` drawn from `dist` ('normal', 'int4' = integers in [-4, 4],
    'full' = whole 8-bit range, 'c_s32' = integers in [-2^20, 2^20])."""
    if dist == "normal":
        x = torch.randn(shape, generator=g, dtype=torch.float32) * std
        if dtype in FMT_MAX:
            return quantize_fp8(x, dtype)
        return x.to(TORCH_DTYPE[dtype])
    if dist == "int4":
        return torch.randint(-4, 5, shape, generator=g).to(TORCH_DTYPE[dtype])
    if dist == "full":
        if dtype == "s8":
            return torch.randint(-128, 128, shape, generator=g).to(torch.int8)
        if dtype == "u8":
            return torch.randint(0, 256, shape, generator=g).to(torch.uint8)
        raise ValueError(dtype)
    if dist == "c_s32":
        return torch.randint(-(1 << 20), (1 << 20) + 1, shape, generator=g).to(torch.int32)
    raise ValueError(dist)


def quantize_fp8(x: torch.Tensor, fmt: str) -> torch.Tensor:
    """Per-tensor scale to the format's maximum, then round-to-nearest-even with
    saturation (input preparation only: the multiply itself takes no scale)."""
    fmax = FMT_MAX[fmt]
    amax = float(x.abs().max())
    s = fmax / amax if amax > 0 else 1.0
    return (x * s).clamp(-fmax, fmax).to(TORCH_DTYPE[fmt])


def apply_mask(A: torch.Tensor, mask: torch.Tensor) -> torch.Tensor:
    """A with the dropped positions set to +0 (bitwise zero)."""
    return torch.where(mask, A, torch.zeros((), dtype=A.dtype))


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw element bits as numpy (uint16 for 16-bit floats, uint8 for FP8/u8, int8 for
    s8, float32 / int32 for the C operand)."""
    t = t.contiguous().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return t.view(torch.uint8).numpy()
    return t.numpy()


def gen_nibbles(shape, g: torch.Generator) -> np.ndarray:
    """Uniform 4-bit patterns (0..15), one per byte: the oracle's 4-bit layout."""
    return torch.randint(0, 16, shape, generator=g).numpy().astype(np.uint8)


def pack4(nibbles) -> np.ndarray:
    """Two 4-bit elements per byte, element 2i in the low nibble (the library's storage)."""
    a = np.asarray(nibbles, dtype=np.uint8)
    return (a[..., 0::2] & 0xF) | ((a[..., 1::2] & 0xF) << 4)


def unpack4(packed) -> np.ndarray:
    """Inverse of pack4: one 4-bit element per byte."""
    a = np.asarray(packed, dtype=np.uint8)
    out = np.empty(a.shape[:-1] + (2 * a.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = a & 0xF
    out[..., 1::2] = a >> 4
    return out


def case(ta: str, tb: str, M: int, N: int, K: int, *, seed: int = 0, tc: str | None = None,
         dist: str = "normal", mask: str = "random", b_dist: str | None = None,
         c_dist: str | None = None) -> dict:
    """Generic seeded case: dense masked A (M x K), its mask, B (K x N), optional C."""
    ga, gb, gc, gm = gen(seed * 4 + 0), gen(seed * 4 + 1), gen(seed * 4 + 2), gen(seed * 4 + 3)
    m = keep_mask(M, K, gm, fixed=(0, 2) if mask == "fixed02" else None)
    A = apply_mask(values((M, K), ta, dist, ga), m)
    B = values((K, N), tb, b_dist or dist, gb)
    C = None
    if tc in ("f32", "f16", "bf16"):
        C = values((M, N), tc, c_dist or "normal", gc)
    elif tc == "s32":
        C = values((M, N), "s32", c_dist or "c_s32", gc)
    return {"A": A, "mask": m, "B": B, "C": C, "ta": ta, "tb": tb, "tc": tc,
            "M": M, "N": N, "K": K}


def fixed_pattern_case() -> dict:
    """The pages' example: one generator seeded 0 draws A (64x128), B (128x64), C (64x64) in order;
    integers in [-4, 4]; fixed positions-0-and-2 pattern."""
    g = gen(0)
    M, N, K = 64, 64, 128
    Araw = torch.randint(-4, 5, (M, K), generator=g).to(torch.float16)
    B = torch.randint(-4, 5, (K, N), generator=g).to(torch.float16)
    C = torch.randint(-4, 5, (M, N), generator=g).to(torch.float32)
    m = keep_mask(M, K, None, fixed=(0, 2))
    return {"A": apply_mask(Araw, m), "mask": m, "B": B, "C": C, "ta": "f16", "tb": "f16",
            "tc": "f32", "M": M, "N": N, "K": K}


def bf16_square(M: int = 4096, N: int = 4096, K: int = 4096) -> dict:
    """bf16, random two-of-four mask, A, B ~ N(0,1), C f32 ~ N(0,1)."""
    m = keep_mask(M, K, gen(3))
    A = apply_mask(values((M, K), "bf16", "normal", gen(0)), m)
    B = values((K, N), "bf16", "normal", gen(1))
    C = values((M, N), "f32", "normal", gen(2))
    return {"A": A, "mask": m, "B": B, "C": C, "ta": "bf16", "tb": "bf16", "tc": "f32",
            "M": M, "N": N, "K": K}


def fp8_square(fmt: str = "e4m3", M: int = 8192, N: int = 8192, K: int = 8192) -> dict:
    """FP8 (same format for A and B), per-tensor scaled N(0,1), random mask, no C."""
    m = keep_mask(M, K, gen(3))
    A = apply_mask(values((M, K), fmt, "normal", gen(0)), m)
    B = values((K, N), fmt, "normal", gen(1))
    return {"A": A, "mask": m, "B": B, "C": None, "ta": fmt, "tb": fmt, "tc": None,
            "M": M, "N": N, "K": K}


def int8_square(ta: str = "s8", M: int = 8192, N: int = 8192, K: int = 8192) -> dict:
    """int8, full 8-bit range (A s8 or u8, B s8), random mask, C s32 in +-2^20."""
    m = keep_mask(M, K, gen(3))
    A = apply_mask(values((M, K), ta, "full", gen(0)), m)
    B = values((K, N), "s8", "full", gen(1))
    C = values((M, N), "s32", "c_s32", gen(2))
    return {"A": A, "mask": m, "B": B, "C": C, "ta": ta, "tb": "s8", "tc": "s32",
            "M": M, "N": N, "K": K}


def llm_layer(N: int = 2048, M: int = 14336, K: int = 4096) -> dict:
    """LLM layer: dense bf16 weight W ~ N(0, 0.02) (no mask: pruned by magnitude on the device)
    and activations X ~ N(0,1)."""
    W = values((M, K), "bf16", "normal", gen(0), std=0.02)
    X = values((K, N), "bf16", "normal", gen(1))
    return {"A": W, "mask": None, "B": X, "C": None, "ta": "bf16", "tb": "bf16", "tc": None,
            "M": M, "N": N, "K": K}
