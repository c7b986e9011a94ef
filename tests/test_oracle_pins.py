"""Pins for the CPU oracle: each test ties it to something other than itself -- a value
the pages print, a library routine, a closed form, an invariant, or brute force on tiny
inputs -- so that a dropped term, a wrong sign or index or a transposed operand fails."""
import itertools
import os

import numpy as np
import pytest
import torch

import inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.strip()
    return out


# --- element decoding: pinned to library conversions over every bit pattern -----------

def test_decode_f16_every_pattern_matches_numpy():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.decode("f16", bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_decode_bf16_every_pattern_matches_torch():
    bits = np.arange(1 << 16, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = oracle.decode("bf16", bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_decode_fp8_every_pattern_matches_torch(fmt, tdt):
    bits = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(bits).view(tdt).double().numpy()
    got = oracle.decode(fmt, bits)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_decode_fp8_closed_forms():
    # OCP FP8: E4M3 max 448 = 1.75 * 2^8, min subnormal 2^-9, no infinity;
    # E5M2 max 57344 = 1.75 * 2^15, min subnormal 2^-16, 0x7c = +inf.
    assert oracle.decode("e4m3", [0x7E])[0] == 448.0
    assert oracle.decode("e4m3", [0x01])[0] == 2.0 ** -9
    assert np.isnan(oracle.decode("e4m3", [0x7F])[0]) and np.isnan(oracle.decode("e4m3", [0xFF])[0])
    assert oracle.decode("e4m3", [0xB8])[0] == -1.0
    assert oracle.decode("e5m2", [0x7B])[0] == 57344.0
    assert oracle.decode("e5m2", [0x01])[0] == 2.0 ** -16
    assert oracle.decode("e5m2", [0x7C])[0] == np.inf
    assert oracle.decode("e5m2", [0x3C])[0] == 1.0


def test_decode_integers():
    b = np.arange(256, dtype=np.uint8)
    assert np.array_equal(oracle.decode("s8", b), b.view(np.int8).astype(np.float64))
    assert np.array_equal(oracle.decode("u8", b), b.astype(np.float64))


def test_decode_4bit_integers_closed_form():
    # the pages' iu4: a 4-bit field, two's complement when the sign flag is set
    n = np.arange(16, dtype=np.uint8)
    assert list(oracle.decode("s4", n)) == [0, 1, 2, 3, 4, 5, 6, 7, -8, -7, -6, -5, -4, -3, -2, -1]
    assert list(oracle.decode("u4", n)) == list(range(16))
    # only the low nibble of the stored byte is the element
    assert oracle.decode("s4", [0xF8])[0] == -8.0 and oracle.decode("u4", [0x37])[0] == 7.0


# --- bf16 rounding: pinned to torch's float32 -> bfloat16 (RNE) and to tie cases -------

def test_round_bf16_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 8)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-40, -3e-39, 3.3e38, -3.4e38])])
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16(x.double().numpy())
    assert np.array_equal(got, ref)


def test_round_bf16_ties_to_even():
    one = 1.0
    ulp = 2.0 ** -7
    # exactly half an ulp above 1.0 -> stays at 1.0 (even); 1.5 ulp -> rounds up to 2 ulp
    assert oracle.round_bf16([one + ulp / 2])[0] == 0x3F80
    assert oracle.round_bf16([one + 1.5 * ulp])[0] == 0x3F82
    assert oracle.round_bf16([one + ulp / 2 + 2.0 ** -30])[0] == 0x3F81
    assert oracle.round_bf16([np.inf])[0] == 0x7F80
    assert oracle.round_bf16([2.0 ** 128])[0] == 0x7F80


# --- f16 rounding (the FP16-accumulate output): pinned to torch's float32 -> float16
# conversion, to the binary16 boundary values and to its own decode

def test_round_f16_matches_torch_on_float32_values():
    g = torch.Generator().manual_seed(6)
    x = torch.randn(200000, generator=g) * torch.exp(torch.randn(200000, generator=g) * 5)
    x = torch.cat([x, torch.tensor([0.0, -0.0, 6e-8, -3e-8, 65504.0, 65519.0, -7e4, 1e-30])])
    ref = x.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_f16(x.double().numpy())
    assert np.array_equal(got, ref)


def test_round_f16_boundaries_and_ties():
    u = 2.0 ** -10                       # ulp of 1.0
    cases = [
        (1.0 + u / 2, 0x3C00),           # half an ulp above 1: ties to even (down)
        (1.0 + 1.5 * u, 0x3C02),         # 1.5 ulp: ties to even (up)
        (1.0 + u / 2 + 2.0 ** -40, 0x3C01),
        (65504.0, 0x7BFF),               # largest finite
        (65519.99, 0x7BFF),
        (65520.0, 0x7C00),               # halfway to 2^16: rounds to infinity
        (-65520.0, 0xFC00),
        (2.0 ** -24, 0x0001),            # smallest subnormal
        (2.0 ** -25, 0x0000),            # half of it: ties to even (zero)
        (1.5 * 2.0 ** -25, 0x0001),
        (1023.5 * 2.0 ** -24, 0x0400),   # between the largest subnormal and 2^-14: even
        (2.0 ** -14, 0x0400),            # smallest normal
        (-0.0, 0x8000),
        (np.inf, 0x7C00),
    ]
    got = oracle.round_f16([c[0] for c in cases])
    assert [int(v) for v in got] == [c[1] for c in cases]
    nan = oracle.round_f16([np.nan])[0]
    assert (nan & 0x7C00) == 0x7C00 and (nan & 0x3FF) != 0


def test_round_f16_inverts_decode():
    bits = np.arange(65536, dtype=np.uint32)
    finite = (bits & 0x7C00) != 0x7C00
    vals = oracle.decode("f16", bits[finite])
    assert np.array_equal(oracle.round_f16(vals), bits[finite].astype(np.uint16))


def test_mma_f64_reads_16_bit_accumulators():
    # B = 0: D is C decoded, for f16 and bf16 C alike
    M, N, K = 3, 8, 32
    values = np.zeros((M, K // 2), dtype=np.uint16)
    index = np.full((M, 1), 0x44444444, dtype=np.uint32)
    B = np.zeros((K, N), dtype=np.uint16)
    for tc in ("f16", "bf16"):
        C = np.arange(M * N, dtype=np.uint16).reshape(M, N) * 37 + 0x3C00
        D, S = oracle.mma_f64(values, index, B, C, "f16", "f16", K, tc=tc)
        assert np.array_equal(D, oracle.decode(tc, C)) and not S.any()


def test_wrap_i32():
    v = np.array([0, 1, -1, 2 ** 31 - 1, 2 ** 31, -(2 ** 31) - 1, 2 ** 32 + 5], dtype=np.int64)
    exp = np.array([0, 1, -1, 2 ** 31 - 1, -(2 ** 31), 2 ** 31 - 1, 5], dtype=np.int32)
    assert np.array_equal(oracle.wrap_i32(v), exp)


# --- the pages' fixed pattern and index literal ----------------------------------------

def test_fixed_pattern_index_literal_0x88():
    fx = _fixture("fixed_pattern_0x88.txt")
    p0, p1 = (int(t) for t in fx["kept_positions"].split())
    byte = int(fx["index_byte_two_groups"], 16)
    word = byte | byte << 8 | byte << 16 | byte << 24
    M, K = 16, 128
    A = np.zeros((M, K), dtype=np.uint16)
    rng = np.random.default_rng(0)
    nz = rng.integers(1, 5, size=(M, K // 4, 2)).astype(np.float16).view(np.uint16)
    A[:, p0::4] = nz[:, :, 0]
    A[:, p1::4] = nz[:, :, 1]
    values, index, flags = oracle.compress(A, "f16", "exact")
    assert not flags.any()
    assert np.all(index == word), hex(int(index[0, 0]))
    assert np.array_equal(values[:, 0::2], A[:, p0::4])
    assert np.array_equal(values[:, 1::2], A[:, p1::4])


def test_fixed_pattern_index_is_all_0x88888888():
    c = inputs.fixed_pattern_case()
    _, index, flags = oracle.compress(inputs.bits(c["A"]), "f16", "mask",
                                      mask=c["mask"].numpy())
    assert not flags.any()
    assert index.shape == (64, 4) and np.all(index == 0x88888888)


# --- compression / decompression round trips -------------------------------------------

@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3", "e5m2", "s8", "u8"])
def test_round_trip_exact_mode(dtype):
    M, K = 24, 96
    g = inputs.gen(11)
    m = inputs.keep_mask(M, K, g)
    dist = "full" if dtype in ("s8", "u8") else "normal"
    A = inputs.values((M, K), dtype, dist, inputs.gen(12))
    # force every kept value non-zero so exact mode sees exactly two per group
    Ab = inputs.bits(A).copy()
    one = inputs.bits(torch.ones(1, dtype=inputs.TORCH_DTYPE[dtype]))[0]
    Ab[Ab == 0] = one
    if dtype in ("f16", "bf16"):
        Ab[Ab == 0x8000] = one
    if dtype in ("e4m3", "e5m2"):
        Ab[Ab == 0x80] = one
    Ab[~m.numpy()] = 0
    values, index, flags = oracle.compress(Ab, dtype, "exact")
    assert not flags.any()
    back = oracle.decompress(values, index, dtype, K)
    assert np.array_equal(back, Ab)
    # the index equals the generating mask, group by group
    _check_index_matches_mask(index, m.numpy())


@pytest.mark.parametrize("dtype", ["s4", "u4"])
def test_round_trip_exact_mode_4bit(dtype):
    M, K = 24, 96
    m = inputs.keep_mask(M, K, inputs.gen(11)).numpy()
    A = inputs.gen_nibbles((M, K), inputs.gen(13))
    A[A == 0] = 1                      # kept values non-zero: exactly two per group
    A[~m] = 0
    values, index, flags = oracle.compress(A, dtype, "exact")
    assert not flags.any()
    assert np.array_equal(oracle.decompress(values, index, dtype, K), A)
    _check_index_matches_mask(index, m)


def _check_index_matches_mask(index, mask):
    M, K = mask.shape
    for i in range(M):
        for g in range(K // 4):
            nib = (int(index[i, g // 8]) >> (4 * (g % 8))) & 0xF
            kept = [p for p in range(4) if mask[i, 4 * g + p]]
            assert nib == (kept[0] | kept[1] << 2), (i, g, nib, kept)


def test_mask_mode_keeps_zero_valued_positions():
    c = inputs.case("f16", "f16", 16, 8, 64, seed=3, dist="int4")
    A = inputs.bits(c["A"])
    m = c["mask"].numpy()
    values, index, flags = oracle.compress(A, "f16", "mask", mask=m)
    assert not flags.any()
    _check_index_matches_mask(index, m)
    assert np.array_equal(oracle.decompress(values, index, "f16", 64), A)


def test_mask_mode_flags_wrong_counts():
    A = np.zeros((1, 8), dtype=np.uint16)
    m = np.array([[1, 1, 1, 0, 1, 0, 0, 0]], dtype=np.uint8)
    _, index, flags = oracle.compress(A, "f16", "mask", mask=m)
    assert flags.tolist() == [[1, 1]]
    # three marked: the two lowest are kept; one marked: filled with the lowest free
    assert int(index[0, 0]) & 0xF == (0 | 1 << 2)
    assert (int(index[0, 0]) >> 4) & 0xF == (0 | 1 << 2)


def test_exact_mode_fill_and_flag_rules():
    h = lambda v: np.float16(v).view(np.uint16)
    A = np.array([[0, 0, 0, 0,               # all zero -> {0,1}
                   0, 0, 0, h(5),            # one non-zero at 3 -> {0,3}
                   0, h(-2), 0, 0,           # one at 1 -> {0,1}
                   h(1), h(2), h(3), 0,      # three -> keep {0,1}, flagged
                   0x8000, h(7), 0, 0x8000,  # -0.0 counts as zero -> {0,1}
                   h(1), 0, 0, h(2),         # exactly two -> {0,3}
                   0, 0, h(4), h(6),         # {2,3}
                   0, h(1), h(1), 0]],       # {1,2}
                 dtype=np.uint16)
    values, index, flags = oracle.compress(A, "f16", "exact")
    nibs = [(int(index[0, 0]) >> (4 * g)) & 0xF for g in range(8)]
    assert nibs == [0x4, 0xC, 0x4, 0x4, 0x4, 0xC, 0xE, 0x9]
    assert flags.tolist() == [[0, 0, 0, 1, 0, 0, 0, 0]]
    assert values[0, 2:4].tolist() == [0, h(5)]
    assert values[0, 4:6].tolist() == [0, h(-2)]


# --- magnitude pruning ------------------------------------------------------------------

def test_magnitude_prune_brute_force_all_small_tuples():
    vals = list(range(-3, 4))
    tuples = list(itertools.product(vals, repeat=4))
    A = np.array(tuples, dtype=np.float16).view(np.uint16).reshape(1, -1)
    values, index, _ = oracle.compress(A, "f16", "magnitude")
    for g, t in enumerate(tuples):
        nib = (int(index[0, g // 8]) >> (4 * (g % 8))) & 0xF
        p0, p1 = nib & 3, nib >> 2
        assert p0 < p1
        kept, dropped = {p0, p1}, set(range(4)) - {p0, p1}
        for d in dropped:
            for k in kept:
                # every dropped |x| <= every kept |x|; at equality the dropped is higher
                assert abs(t[d]) < abs(t[k]) or (abs(t[d]) == abs(t[k]) and d > k), (t, nib)
        assert values[0, 2 * g] == A[0, 4 * g + p0] and values[0, 2 * g + 1] == A[0, 4 * g + p1]


def test_magnitude_prune_brute_force_all_s4_groups():
    # every group of four 4-bit two's-complement values (16^4): dropped |x| <= kept |x|,
    # ties drop the higher position; -8 has magnitude 8, the largest
    tuples = np.array(list(itertools.product(range(16), repeat=4)), dtype=np.uint8)
    A = tuples.reshape(1, -1)
    values, index, _ = oracle.compress(A, "s4", "magnitude")
    mag = np.abs(oracle.decode("s4", tuples))
    nib = (index[0][np.arange(len(tuples)) // 8] >> (4 * (np.arange(len(tuples)) % 8))) & 0xF
    p0, p1 = nib & 3, nib >> 2
    assert np.all(p0 < p1)
    for g in range(len(tuples)):
        kept = {int(p0[g]), int(p1[g])}
        for d in set(range(4)) - kept:
            for k in kept:
                assert mag[g, d] < mag[g, k] or (mag[g, d] == mag[g, k] and d > k)
    assert np.array_equal(values[0, 0::2], A[0, 4 * np.arange(len(tuples)) + p0])


def test_magnitude_prune_matches_sorted_selection_bf16():
    W = inputs.values((32, 256), "bf16", "normal", inputs.gen(0), std=0.02)
    Wb = inputs.bits(W)
    Wd = W.double().numpy()
    _, index, _ = oracle.compress(Wb, "bf16", "magnitude")
    for i in range(32):
        for g in range(64):
            grp = Wd[i, 4 * g:4 * g + 4]
            order = sorted(range(4), key=lambda p: (-abs(grp[p]), p))
            want = sorted(order[:2])
            nib = (int(index[i, g // 8]) >> (4 * (g % 8))) & 0xF
            assert [nib & 3, nib >> 2] == want


# --- the product: brute force, identity, library dense product --------------------------

def test_all_six_patterns_brute_force_dense_product():
    rng = np.random.default_rng(1)
    for M, N, K in [(1, 1, 4), (3, 5, 32), (8, 8, 64), (5, 7, 36)]:
        for pat in inputs.PATTERNS:
            m = np.zeros((M, K), dtype=bool)
            for p in pat:
                m[:, p::4] = True
            Ai = np.where(m, rng.integers(-4, 5, size=(M, K)), 0)
            Bi = rng.integers(-4, 5, size=(K, N))
            Ci = rng.integers(-4, 5, size=(M, N))
            A = Ai.astype(np.float16).view(np.uint16)
            B = Bi.astype(np.float16).view(np.uint16)
            values, index, flags = oracle.compress(A, "f16", "mask", mask=m)
            D, S = oracle.mma_f64(values, index, B, Ci.astype(np.float32), "f16", "f16", K)
            want = Ci + Ai @ Bi  # dense(A_masked) @ B + C, exact integers
            assert np.array_equal(D, want.astype(np.float64)), (M, N, K, pat)
            assert np.array_equal(S, (np.abs(Ai) @ np.abs(Bi)).astype(np.float64))


def test_identity_B_gives_expanded_A_plus_C():
    # the pages' verification idiom: B = I, so the product is A itself
    c = inputs.case("bf16", "bf16", 32, 64, 64, seed=7, tc="f32")
    A = inputs.bits(c["A"])
    values, index, _ = oracle.compress(A, "bf16", "mask", mask=c["mask"].numpy())
    eye = torch.eye(64, dtype=torch.bfloat16)
    D, _ = oracle.mma_f64(values, index, inputs.bits(eye), c["C"].numpy(), "bf16", "bf16", 64)
    want = c["A"].double().numpy() + c["C"].double().numpy()
    assert np.array_equal(D, want)


@pytest.mark.parametrize("ta,tb", [("f16", "f16"), ("bf16", "bf16"), ("e4m3", "e4m3"),
                                   ("e5m2", "e5m2")])
def test_mma_f64_matches_library_dense_product(ta, tb):
    c = inputs.case(ta, tb, 40, 24, 96, seed=2, tc="f32")
    values, index, _ = oracle.compress(inputs.bits(c["A"]), ta, "mask", mask=c["mask"].numpy())
    D, S = oracle.mma_f64(values, index, inputs.bits(c["B"]), c["C"].numpy(), ta, tb, 96)
    Ad = c["A"].double().numpy()
    Bd = c["B"].double().numpy()
    want = c["C"].double().numpy() + Ad @ Bd
    assert np.allclose(D, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(S, np.abs(Ad) @ np.abs(Bd), rtol=1e-12, atol=0)


@pytest.mark.parametrize("ta", ["s8", "u8"])
def test_mma_i64_matches_integer_dense_product(ta):
    c = inputs.case(ta, "s8", 33, 17, 128, seed=4, dist="full", tc="s32")
    A = inputs.bits(c["A"])
    values, index, _ = oracle.compress(A, ta, "mask", mask=c["mask"].numpy())
    D = oracle.mma_i64(values, index, inputs.bits(c["B"]), c["C"].numpy(), ta, "s8", 128)
    want = c["C"].numpy().astype(np.int64) + A.astype(np.int64) @ c["B"].numpy().astype(np.int64)
    assert np.array_equal(D, want)


def test_integer_extremes_exact():
    # every kept a = -128 (or 255 unsigned) and every b = -128: the largest |a*b| terms
    M, N, K = 4, 4, 64
    m = inputs.keep_mask(M, K, inputs.gen(9)).numpy()
    for ta, aval in (("s8", -128), ("u8", 255)):
        Ai = np.where(m, aval, 0)
        A = Ai.astype(np.int64).astype(np.uint8 if ta == "u8" else np.int8)
        Bi = np.full((K, N), -128)
        values, index, _ = oracle.compress(A, ta, "mask", mask=m)
        D = oracle.mma_i64(values, index, Bi.astype(np.int8), None, ta, "s8", K)
        assert np.array_equal(D, Ai @ Bi)


@pytest.mark.parametrize("ta", ["s4", "u4"])
def test_mma_i64_4bit_matches_integer_dense_product(ta):
    M, N, K = 33, 17, 128
    m = inputs.keep_mask(M, K, inputs.gen(21)).numpy()
    A = inputs.gen_nibbles((M, K), inputs.gen(22))
    A[~m] = 0
    B = inputs.gen_nibbles((K, N), inputs.gen(23))
    C = np.random.default_rng(24).integers(-2**20, 2**20, (M, N)).astype(np.int32)
    values, index, _ = oracle.compress(A, ta, "mask", mask=m)
    D = oracle.mma_i64(values, index, B, C, ta, "s4", K)
    # the same product written with numpy's own 4-bit decoding
    Ai = A.astype(np.int64) - (16 * (A >= 8) if ta == "s4" else 0)
    Bi = B.astype(np.int64) - 16 * (B >= 8)
    assert np.array_equal(D, C.astype(np.int64) + Ai @ Bi)
    # extremes: every kept a at -8 (or 15) and every b = -8
    Ae = np.where(m, 8 if ta == "s4" else 15, 0).astype(np.uint8)
    v2, i2, _ = oracle.compress(Ae, ta, "mask", mask=m)
    D2 = oracle.mma_i64(v2, i2, np.full((K, N), 8, np.uint8), None, ta, "s4", K)
    aval = -8 if ta == "s4" else 15
    assert np.array_equal(D2, (m * aval).astype(np.int64) @ np.full((K, N), -8))


def test_row_subset_equals_full_rows():
    c = inputs.case("bf16", "bf16", 50, 16, 64, seed=8, tc="f32")
    values, index, _ = oracle.compress(inputs.bits(c["A"]), "bf16", "mask", mask=c["mask"].numpy())
    Df, Sf = oracle.mma_f64(values, index, inputs.bits(c["B"]), c["C"].numpy(), "bf16", "bf16", 64)
    rows = [0, 7, 49, 13]
    Dr, Sr = oracle.mma_f64(values, index, inputs.bits(c["B"]), c["C"].numpy(), "bf16", "bf16", 64,
                            rows=rows)
    assert np.array_equal(Dr, Df[rows]) and np.array_equal(Sr, Sf[rows])


def test_tolerance_rejects_a_transposed_operand():
    # a plausible mistake (B used transposed) must fall outside the float tolerance
    c = inputs.case("bf16", "bf16", 32, 32, 32, seed=10, tc="f32")
    values, index, _ = oracle.compress(inputs.bits(c["A"]), "bf16", "mask", mask=c["mask"].numpy())
    D, S = oracle.mma_f64(values, index, inputs.bits(c["B"]), c["C"].numpy(), "bf16", "bf16", 32)
    bad = c["C"].double().numpy() + c["A"].double().numpy() @ c["B"].double().numpy().T
    assert not oracle.tolerance_ok(bad, D, S).all()
    assert oracle.tolerance_ok(D + 1e-9 * S, D, S).all()
