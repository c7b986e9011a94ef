"""The sparse GEMM (tcgen05.mma.sp) against the oracle: small ragged cases span several
tiles and every tail; the workload sizes run at full size in the bench's launch
configuration and are compared on sampled rows."""
import numpy as np
import pytest
import torch

import inputs
import oracle
import structured_sparse_matrix_gb300 as sp
from parity import check_float, dev, gpu_compress, run_case, sample_rows, tile_quarter_rows

pytestmark = pytest.mark.gpu

FLOAT_TYPES = ["f16", "bf16", "e4m3", "e5m2"]


def test_fixed_pattern_bit_exact():
    # integer-valued f16 inputs: every partial sum is a small integer, so D is exact
    c = inputs.fixed_pattern_case()
    Dg, Dref, _ = run_case(c, mode="mask", check=False)
    assert np.array_equal(Dg.astype(np.float64), Dref)


@pytest.mark.parametrize("ta", FLOAT_TYPES)
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 192, 320), (257, 64, 96),
                                   (64, 304, 512), (1, 16, 32), (384, 400, 1056),
                                   (200, 16, 384), (257, 32, 1056), (130, 48, 256)])
def test_small_ragged_shapes(ta, M, N, K):
    c = inputs.case(ta, ta, M, N, K, seed=M + N + K, tc="f32")
    run_case(c, mode="mask")


@pytest.mark.parametrize("ta", ["f16", "bf16"])
@pytest.mark.parametrize("M,N,K", [(130, 24, 256), (64, 8, 128), (300, 16, 2080),
                                   (130, 16, 480), (129, 32, 4256)])
def test_skinny_outputs(ta, M, N, K):
    # N <= 32 runs on 128 x 32 tiles that stage only the B columns below N; 16-bit
    # operands take 256 dense K (two boxes of A, eight MMAs) per stage, so K = 480 and
    # 4256 end on a stage whose second box is partly past K
    c = inputs.case(ta, ta, M, N, K, seed=M + N + K, tc="f32")
    run_case(c, mode="mask")
    run_case(dict(c, C=None, tc=None), mode="mask", out_dtype=torch.bfloat16)


@pytest.mark.parametrize("ta", FLOAT_TYPES)
def test_no_C_and_bf16_output(ta):
    c = inputs.case(ta, ta, 300, 272, 384, seed=12, tc=None)
    run_case(c, mode="mask", out_dtype=torch.float32)
    run_case(c, mode="mask", out_dtype=torch.bfloat16)


@pytest.mark.parametrize("ta,tb", [("e4m3", "e5m2"), ("e5m2", "e4m3")])
@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (200, 304, 512), (130, 16, 768),
                                   (384, 400, 1280)])
def test_mixed_fp8_operands(ta, tb, M, N, K):
    # kind::f8f6f4 takes separate A and B types: E4M3 x E5M2 and E5M2 x E4M3
    c = inputs.case(ta, tb, M, N, K, seed=M + 3 * N + K, tc="f32")
    run_case(c, mode="mask")
    run_case(dict(c, C=None, tc=None), mode="mask", out_dtype=torch.bfloat16)


@pytest.mark.parametrize("ta", ["f16", "e4m3"])
def test_every_single_pattern(ta):
    # one pattern everywhere, for each of the six: exercises every metadata nibble value
    for pat in inputs.PATTERNS:
        M, N, K = 128, 128, 256
        g = inputs.gen(100)
        A = inputs.values((M, K), ta, "normal", g)
        m = inputs.keep_mask(M, K, None, fixed=pat)
        c = {"A": inputs.apply_mask(A, m), "mask": m,
             "B": inputs.values((K, N), ta, "normal", inputs.gen(101)),
             "C": None, "ta": ta, "tb": ta, "tc": None, "M": M, "N": N, "K": K}
        run_case(c, mode="mask")


@pytest.mark.parametrize("ta", ["bf16", "e5m2"])
def test_padded_leading_dimensions_and_ragged_N(ta):
    # N = 300 is not a legal row pitch for 8-bit B; padded buffers (ld = 320) carry it
    M, N, K, ld = 160, 300, 256, 320
    c = inputs.case(ta, ta, M, N, K, seed=40, tc="f32")
    Bp = torch.zeros((K, ld), dtype=c["B"].dtype)
    Bp[:, :N] = c["B"]
    Cp = torch.zeros((M, ld), dtype=torch.float32)
    Cp[:, :N] = c["C"]
    Dp = torch.full((M, ld), 7.0, dtype=torch.float32, device="cuda")
    values, index = sp.compress(dev(c["A"]), mode="mask", mask=dev(c["mask"]))
    meta = sp.meta_prepare(index, c["A"].dtype, M, K)
    sp.mma(values, meta, Bp.cuda()[:, :N], Cp.cuda()[:, :N], out=Dp[:, :N])
    torch.cuda.synchronize()
    v, i, _ = oracle.compress(inputs.bits(c["A"]), ta, "mask", mask=c["mask"].numpy())
    R, S = oracle.mma_f64(v, i, inputs.bits(c["B"]), c["C"].numpy(), ta, ta, K)
    Dh = Dp.cpu().numpy()
    check_float(Dh[:, :N], R, S, False, "padded")
    assert np.all(Dh[:, N:] == 7.0), "wrote past N"


@pytest.mark.parametrize("ta,tb,M,N,K", [("bf16", "bf16", 200, 304, 384),   # pair tiles
                                        ("f16", "f16", 130, 96, 256),     # single tiles
                                        ("e4m3", "e5m2", 257, 16, 512),   # narrow tiles
                                        ("bf16", "bf16", 257, 16, 480),   # narrow, 256-K stages
                                        ("bf16", "bf16", 64, 272, 0)])    # K = 0: D = C
def test_strided_batch(ta, tb, M, N, K):
    # four problems of one shape in one launch, each against the oracle, and bit for bit
    # equal to four single calls (same tiles, same accumulation order)
    cases = [inputs.case(ta, tb, M, N, K, seed=500 + i, tc="f32") for i in range(4)]
    Kc = max(K, 32)
    vals, metas = [], []
    for c in cases:
        if K > 0:
            v, ix = sp.compress(dev(c["A"]), mode="mask", mask=dev(c["mask"]))
            vals.append(v)
            metas.append(sp.meta_prepare(ix, c["A"].dtype, M, K))
        else:
            vals.append(torch.zeros((M, Kc // 2), dtype=c["A"].dtype, device="cuda"))
            metas.append(torch.zeros(16, dtype=torch.uint8, device="cuda"))
    V = torch.stack(vals)
    MT = torch.stack(metas)
    Bs = torch.stack([dev(c["B"]) for c in cases])
    Cs = torch.stack([dev(c["C"]) for c in cases])
    D = sp.mma_batched(V, MT, Bs, Cs)
    singles = [sp.mma(vals[i], metas[i], Bs[i], Cs[i]) for i in range(4)]
    torch.cuda.synchronize()
    for i, c in enumerate(cases):
        assert torch.equal(D[i], singles[i]), f"problem {i} differs from the single call"
        if K == 0:
            assert torch.equal(D[i], Cs[i])
            continue
        v, ix, _ = oracle.compress(inputs.bits(c["A"]), ta, "mask", mask=c["mask"].numpy())
        R, S = oracle.mma_f64(v, ix, inputs.bits(c["B"]), c["C"].numpy(), ta, tb, K)
        check_float(D[i].cpu().numpy(), R, S, False, f"batched problem {i}")


def test_identity_B_returns_A_plus_C():
    # the pages' verification idiom: with B = I the product is A itself
    M, K = 256, 256
    c = inputs.case("bf16", "bf16", M, K, K, seed=31, tc="f32")
    c["B"] = torch.eye(K, dtype=torch.bfloat16)
    values, index = sp.compress(dev(c["A"]), mode="mask", mask=dev(c["mask"]))
    meta = sp.meta_prepare(index, torch.bfloat16, M, K)
    D = sp.mma(values, meta, dev(c["B"]), dev(c["C"]))
    torch.cuda.synchronize()
    want = (c["A"].float() + c["C"]).numpy()
    assert np.array_equal(D.cpu().numpy(), want)


def test_K_zero_gives_C():
    M, N = 130, 72
    C = torch.randn(M, N, generator=inputs.gen(2)).cuda()
    B = torch.empty((0, N), dtype=torch.float16, device="cuda")
    values = torch.empty((M, 0), dtype=torch.float16, device="cuda")
    meta = torch.empty(16, dtype=torch.uint8, device="cuda")
    D = sp.mma(values, meta, B, C)
    torch.cuda.synchronize()
    assert torch.equal(D, C)


def test_matmul_through_sparse_matrix_object():
    c = inputs.case("f16", "f16", 192, 64, 128, seed=3, dist="int4", tc="f32", c_dist="int4")
    W = sp.SparseMatrix.from_dense(dev(c["A"]), mode="mask", mask=dev(c["mask"]))
    D = W.matmul(dev(c["B"]), dev(c["C"]))
    back = W.to_dense()
    torch.cuda.synchronize()
    assert torch.equal(back.cpu(), c["A"])
    want = c["C"].double() + c["A"].double() @ c["B"].double()
    assert np.array_equal(D.cpu().double().numpy(), want.numpy())


def test_bounded_wait_gives_up_and_context_survives():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = sp.lib().sp24_diag_wait_timeout(sp._ptr(status), 20_000_000, sp._stream())
    assert rc == 0
    torch.cuda.synchronize()
    assert status.item() & sp.DEV_TIMEOUT
    # the context is still usable
    x = torch.ones(4, device="cuda") * 2
    assert float(x.sum()) == 8.0


@pytest.mark.parametrize("ta,N", [("bf16", 256),   # CTA pair, 256 x 256 tiles
                                  ("bf16", 96),    # CTA pair, 256 x 128 tiles
                                  ("e4m3", 96),    # one CTA, 128 x 128 tiles
                                  ("bf16", 16)])   # one CTA, 128 x 32 tiles
def test_gemm_gives_up_when_operands_never_arrive(ta, N):
    """The product kernel itself, with its TMA producer issuing nothing: the MMA thread's
    bounded wait gives up, every role stops, SP24_DEV_TIMEOUT is set, and the context stays
    usable -- a following ordinary product still matches the oracle."""
    M, K = 256, 512
    c = inputs.case(ta, ta, M, N, K, seed=11)
    values, index, _ = gpu_compress(c, "mask")
    meta = sp.meta_prepare(index, c["A"].dtype, M, K)
    B = dev(c["B"])
    D = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = sp.lib().sp24_diag_mma_stall(sp.DTYPE_CODES[c["A"].dtype], M, N, K, sp._ptr(values),
                                      values.stride(0), sp._ptr(meta), sp._ptr(B), B.stride(0),
                                      sp._ptr(D), D.stride(0), 20_000_000, sp._ptr(status),
                                      sp._stream())
    assert rc == 0
    torch.cuda.synchronize()
    assert status.item() & sp.DEV_TIMEOUT
    assert torch.all(D == 7.0)  # the epilogue never ran
    # the context is still usable: the same problem through sp24_mma matches the oracle
    run_case(c, mode="mask")


# ---- full-size workloads, compared on sampled rows --------------------------------------

def test_full_size_bf16_4096():
    # every element of the 4096^3 product against the oracle (about 20 s of oracle time)
    c = inputs.bf16_square()
    run_case(c, mode="mask")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_full_size_fp8_8192(fmt):
    c = inputs.fp8_square(fmt)
    run_case(c, mode="mask", rows=tile_quarter_rows(c["M"]))


@pytest.mark.parametrize("N", [16, 128, 2048])
def test_llm_layer(N):
    # N = 16 and 128: every row; N = 2048: sampled rows
    c = inputs.llm_layer(N=N)
    run_case(c, mode="magnitude", out_dtype=torch.bfloat16,
             rows=sample_rows(c["M"]) if N > 128 else None)


# ---- 8-bit integers: exact, through the bf16 path with chunked int32 accumulation ----------

@pytest.mark.parametrize("ta", ["s8", "u8"])
@pytest.mark.parametrize("M,N,K", [(128, 128, 128), (200, 192, 1056), (33, 48, 2080),
                                   (257, 272, 320)])
def test_int8_small_ragged_exact(ta, M, N, K):
    c = inputs.case(ta, "s8", M, N, K, seed=M + K, dist="full", tc="s32")
    run_case(c, mode="mask", out_dtype=torch.int32)


@pytest.mark.parametrize("ta,aval", [("s8", -128), ("u8", 255)])
def test_int8_extreme_values_many_chunks(ta, aval):
    # every kept a at its extreme and every b = -128: the largest |a b| terms; K = 4096
    # spans four 1024-K chunks and each output is -2048 * |a| * 128, far beyond 2^24
    M, N, K = 128, 144, 4096
    m = inputs.keep_mask(M, K, inputs.gen(5))
    Ai = torch.where(m, torch.full((M, K), aval), torch.zeros((M, K), dtype=torch.long))
    A = Ai.to(torch.int8 if ta == "s8" else torch.uint8)
    B = torch.full((K, N), -128, dtype=torch.int8)
    C = torch.full((M, N), -(1 << 20), dtype=torch.int32)
    c = {"A": A, "mask": m, "B": B, "C": C, "ta": ta, "tb": "s8", "tc": "s32",
         "M": M, "N": N, "K": K}
    Dg, Dref, _ = run_case(c, mode="mask", out_dtype=torch.int32)
    assert int(np.abs(Dref).max()) > (1 << 24)


def test_int8_wraps_like_int32():
    # C near the int32 limit: the result wraps modulo 2^32 (no clamp)
    M, N, K = 128, 128, 64
    m = inputs.keep_mask(M, K, None, fixed=(0, 1))
    A = torch.where(m, torch.full((M, K), 127), torch.zeros((M, K), dtype=torch.long)).to(torch.int8)
    B = torch.full((K, N), 127, dtype=torch.int8)
    C = torch.full((M, N), 2**31 - 1000, dtype=torch.int32)
    c = {"A": A, "mask": m, "B": B, "C": C, "ta": "s8", "tb": "s8", "tc": "s32",
         "M": M, "N": N, "K": K}
    Dg, Dref, _ = run_case(c, mode="mask", out_dtype=torch.int32)
    assert int(Dref.max()) > 2**31 - 1 and int(Dg.min()) < 0


@pytest.mark.parametrize("ta", ["s8", "u8"])
def test_full_size_int8_8192(ta):
    c = inputs.int8_square(ta)
    run_case(c, mode="mask", out_dtype=torch.int32, rows=tile_quarter_rows(c["M"]))


# ---- 16-bit C and D: the FP16- / BF16-accumulate forms and mixed accumulator types -------

@pytest.mark.parametrize("ta,tc,out", [("f16", "f16", torch.float16),
                                       ("bf16", "bf16", torch.bfloat16),
                                       ("f16", "f32", torch.float16),
                                       ("bf16", "f16", torch.float32),
                                       ("e4m3", "bf16", torch.float16),
                                       ("e5m2", "f16", torch.bfloat16)])
@pytest.mark.parametrize("M,N,K", [(200, 16, 384), (130, 96, 256), (257, 272, 1056)])
def test_16bit_accumulator_forms(ta, tc, out, M, N, K):
    # narrow (N <= 32), single (N <= 128) and pair (N > 128) variants, ragged M and N; FP8
    # operands are small integers (a tensor scaled to the FP8 maximum would overflow f16)
    c = inputs.case(ta, ta, M, N, K, seed=M + N, tc=tc,
                    dist="int4" if ta in ("e4m3", "e5m2") else "normal")
    run_case(c, mode="mask", out_dtype=out)


def test_f16_accumulate_full_size_sampled():
    # the FP16-accumulate form (f16 A, B, C, D) at 4096^3, checked on sampled rows
    c = inputs.case("f16", "f16", 4096, 4096, 4096, seed=77, tc="f16")
    run_case(c, mode="mask", out_dtype=torch.float16, rows=sample_rows(4096))


def test_f16_output_overflows_to_infinity():
    # a result beyond the binary16 range rounds to +-inf, as the oracle's rounding does
    # every kept a = 4 and b = +-4 by column: the sums are +-1024 (K = 128), C = +-65000
    # with the same sign, so every exact result is +-66024 (beyond 65519.99...)
    M, N, K = 128, 64, 128
    c = inputs.case("f16", "f16", M, N, K, seed=4, tc="f16", dist="int4")
    c["A"] = torch.where(c["mask"], torch.tensor(4.0), torch.tensor(0.0)).to(torch.float16)
    sign = torch.where(torch.arange(N) % 2 == 0, -1.0, 1.0)
    c["B"] = (4.0 * sign).expand(K, N).contiguous().to(torch.float16)
    c["C"] = (65000.0 * sign).expand(M, N).contiguous().to(torch.float16)
    Dg, Dref, _ = run_case(c, mode="mask", out_dtype=torch.float16)
    assert np.all(np.isinf(Dg)) and np.all(np.sign(Dg) == sign.numpy())


# ---- the product on the image written by the fused compression pass ---------------------

@pytest.mark.parametrize("ta,tc,out", [("bf16", "f32", torch.float32),
                                       ("e4m3", None, torch.bfloat16),
                                       ("s8", "s32", torch.int32)])
@pytest.mark.parametrize("M,N,K", [(200, 16, 384), (257, 272, 1056)])
def test_product_on_fused_image(ta, tc, out, M, N, K):
    c = inputs.case(ta, "s8" if ta == "s8" else ta, M, N, K, seed=M + 3, tc=tc,
                    dist="full" if ta == "s8" else "normal")
    run_case(c, mode="mask", out_dtype=out, fused=True)


def test_bf16_4096_through_the_fused_pass():
    c = inputs.bf16_square()
    run_case(c, mode="mask", rows=sample_rows(c["M"]), fused=True)


# ---- CUDA graphs: the calls are stream-ordered and allocation-free, so they capture --------

def test_graph_capture_replays_the_eager_result():
    M, N, K = 1000, 200, 1024
    c = inputs.case("bf16", "bf16", M, N, K, seed=12, tc="f32")
    A, mask, B, C = c["A"].cuda(), c["mask"].cuda().to(torch.uint8), c["B"].cuda(), c["C"].cuda()
    values = torch.empty((M, K // 2), dtype=torch.bfloat16, device="cuda")
    index = torch.empty((M, K // 32), dtype=torch.int32, device="cuda")
    meta = torch.empty(sp.meta_bytes(torch.bfloat16, M, K), dtype=torch.uint8, device="cuda")
    D = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L = sp.lib()

    def step():
        st = sp._stream(torch.cuda.current_stream())
        assert L.sp24_compress_meta(1, M, K, sp._ptr(A), K, sp._ptr(mask), K, 1, sp._ptr(values),
                                    K // 2, sp._ptr(index), K // 32, sp._ptr(meta), None, st) == 0
        assert L.sp24_mma(1, 1, 6, 6, M, N, K, sp._ptr(values), K // 2, sp._ptr(meta),
                          sp._ptr(B), N, sp._ptr(C), N, sp._ptr(D), N, None, 0, None, st) == 0

    step()  # eager (also sets up the kernels' attributes before capture)
    torch.cuda.synchronize()
    eager = D.clone()
    D.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    D.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(D, eager)
    rows = sample_rows(M)
    v_ref, i_ref, _ = oracle.compress(inputs.bits(c["A"]), "bf16", "mask", mask=c["mask"].numpy())
    Dref, S = oracle.mma_f64(v_ref, i_ref, inputs.bits(c["B"]), c["C"].numpy(), "bf16", "bf16", K,
                             rows=rows)
    check_float(D.cpu().numpy()[rows], Dref, S, False, "graph replay")


# ---- large extents: many row tiles, very long K ------------------------------------------

@pytest.mark.parametrize("ta,M,N,K", [("bf16", 200_000, 16, 64),      # 1563 narrow tiles
                                      ("bf16", 128, 128, 131_072),    # 1024 K stages
                                      ("e4m3", 300, 48, 65_536)])     # 256 FP8 stages
def test_large_extents(ta, M, N, K):
    c = inputs.case(ta, ta, M, N, K, seed=M % 97, tc="f32",
                    dist="int4" if ta == "e4m3" else "normal")
    run_case(c, mode="mask", rows=sample_rows(M)[::7], fused=True)


def test_int8_long_k_exact():
    # K = 65536: 32 chunks of the s8 x s8 integer accumulation, every product at its extreme
    M, N, K = 256, 64, 65_536
    m = inputs.keep_mask(M, K, inputs.gen(3))
    A = torch.where(m, torch.full((M, K), -128), torch.zeros((M, K), dtype=torch.long)).to(torch.int8)
    B = torch.full((K, N), -128, dtype=torch.int8)
    C = torch.zeros((M, N), dtype=torch.int32)
    c = {"A": A, "mask": m, "B": B, "C": C, "ta": "s8", "tb": "s8", "tc": "s32",
         "M": M, "N": N, "K": K}
    Dg, Dref, _ = run_case(c, mode="mask", out_dtype=torch.int32, rows=np.arange(0, M, 17))
    assert np.all(Dref == (K // 2) * 16384)   # 2^29: far beyond 2^24, exact


# ---- grouped products: problems of different shapes in one launch -----------------------

def _grouped_case(ta, shapes, tc, out, seed):
    items, refs = [], []
    for i, (M, N, K) in enumerate(shapes):
        c = inputs.case(ta, ta, M, N, K, seed=seed + i, tc=tc,
                        dist="int4" if ta in ("e4m3", "e5m2") else "normal")
        values, index, meta = sp.compress_meta(c["A"].cuda(), mode="mask", mask=c["mask"].cuda())
        items.append((values, meta, c["B"].cuda(), None if c["C"] is None else c["C"].cuda()))
        refs.append(c)
    D = sp.mma_grouped(items, out_dtype=out)
    torch.cuda.synchronize()
    for c, Dg in zip(refs, D):
        M, N, K = c["M"], c["N"], c["K"]
        v_ref, i_ref, _ = oracle.compress(inputs.bits(c["A"]), ta, "mask", mask=c["mask"].numpy())
        rows = sample_rows(M)
        Dref, S = oracle.mma_f64(v_ref, i_ref, inputs.bits(c["B"]),
                                 None if c["C"] is None else inputs.bits(c["C"]), ta, ta, K,
                                 tc=tc or "f32", rows=rows)
        from parity import OUT_KIND
        check_float(Dg.float().cpu().numpy()[rows], Dref, S, OUT_KIND[out],
                    f"grouped {ta} {M}x{N}x{K}")


@pytest.mark.parametrize("ta,shapes,tc,out", [
    # widest N > 128: 256 x 256 pair tiles for all
    ("bf16", [(300, 200, 352), (128, 64, 128), (513, 136, 1056), (64, 8, 64)], "f32",
     torch.float32),
    # widest N <= 32: narrow tiles, each problem its own MMA N
    ("e4m3", [(1000, 16, 512), (200, 32, 256), (64, 32, 1024)], None, torch.bfloat16),
    # the same with 16-bit operands (256-K stages; each problem its own ragged last stage)
    ("bf16", [(500, 16, 480), (130, 24, 256), (64, 8, 96)], "f32", torch.float32),
    # 32 < widest N <= 128, 16-bit: 256 x 128 pair tiles; FP8: 128 x 128 single tiles
    ("f16", [(700, 104, 384), (129, 40, 128), (256, 128, 2048)], "f16", torch.float16),
    ("e5m2", [(700, 112, 512), (129, 48, 256)], "f32", torch.float32),
])
def test_grouped_shapes(ta, shapes, tc, out):
    _grouped_case(ta, shapes, tc, out, seed=len(shapes))


def test_grouped_many_problems_and_empty_ones():
    # 40 problems (two launches of 32 and 8), two of them empty
    shapes = [(64 + 16 * (i % 5), 16 * (1 + i % 3), 128 * (1 + i % 2)) for i in range(38)]
    _grouped_case("bf16", shapes, "f32", torch.float32, seed=100)
    values = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    meta = torch.empty(16, dtype=torch.uint8, device="cuda")
    B = torch.zeros((128, 16), dtype=torch.bfloat16, device="cuda")
    D = sp.mma_grouped([(values, meta, B, None)])
    assert D[0].shape == (0, 16)


# ---- the product on the canonical index itself (no image) ---------------------------------

@pytest.mark.parametrize("ta,tb,tc,out,M,N,K", [
    ("bf16", "bf16", "f32", torch.float32, 200, 16, 352),    # narrow tiles, ragged M and K
    ("f16", "f16", "f32", torch.float32, 150, 24, 480),      # narrow: last stage's 2nd box
    ("f16", "f16", None, torch.bfloat16, 130, 96, 160),      # 256 x 128 pair tiles
    ("bf16", "bf16", "bf16", torch.float32, 257, 272, 1056),  # 256 x 256 pair tiles
    ("e4m3", "e4m3", None, torch.float32, 131, 80, 544),     # FP8, 128 x 128 tiles
    ("e5m2", "e4m3", "f32", torch.float32, 300, 304, 800),   # FP8 pair, stage tail
    ("e4m3", "e4m3", None, torch.bfloat16, 64, 32, 256),     # FP8 narrow tiles
    ("s8", "s8", "s32", torch.int32, 190, 144, 1088),        # exact integers (16-bit layout)
    ("u8", "s8", "s32", torch.int32, 130, 272, 2080),        # u8 x s8: 1024-K exact chunks
])
def test_product_reads_the_canonical_index(ta, tb, tc, out, M, N, K):
    c = inputs.case(ta, tb, M, N, K, seed=M + N, tc=tc,
                    dist="full" if ta in ("s8", "u8") else "normal")
    run_case(c, mode="mask", out_dtype=out, by_index=True)


@pytest.mark.parametrize("N", [64, 16])
def test_canonical_index_with_a_padded_pitch(N):
    # a pitch of K/32 + 3 words: the writers load the words one by one
    M, K = 250, 480
    c = inputs.case("bf16", "bf16", M, N, K, seed=17, tc="f32")
    values, index, _ = gpu_compress(c, "mask")
    wide = torch.full((M, K // 32 + 3), -1, dtype=torch.int32, device="cuda")
    wide[:, :K // 32] = index
    B, C = dev(c["B"]), dev(c["C"])
    D_idx = sp.mma_index(values, wide[:, :K // 32], B, C)
    D_img = sp.mma(values, sp.meta_prepare(index, torch.bfloat16, M, K), B, C)
    torch.cuda.synchronize()
    assert torch.equal(D_idx.view(torch.uint8), D_img.view(torch.uint8))


def test_llm_layer_through_the_index():
    c = inputs.llm_layer(16)
    run_case(c, mode="magnitude", out_dtype=torch.bfloat16, rows=sample_rows(c["M"]),
             by_index=True)


# ---- products back to back on one stream, the second reading the first's output --------

@pytest.mark.parametrize("N", [16, 288])          # narrow tiles; 256 x 256 pair tiles
@pytest.mark.parametrize("graph", [False, True])
def test_layers_chained_on_one_stream(N, graph):
    # Y1 = W1 X, then Y2 = W2 Y1 + Y0, enqueued back to back with no synchronisation: the
    # second product takes the first's output as its B.  Products overlap their launch and
    # set-up with the kernel before them and fetch their first stages into L2 early, so this
    # checks that the second one reads Y1 only once the first has written all of it (Y1
    # and Y2 start out holding huge values, which would show up in any early read).
    M1, K1, M2 = 384, 512, 320
    c1 = inputs.case("bf16", "bf16", M1, N, K1, seed=N + 1, tc=None)
    c2 = inputs.case("bf16", "bf16", M2, N, M1, seed=N + 2, tc="f32")
    v1, i1, s1 = gpu_compress(c1, "mask")
    v2, i2, s2 = gpu_compress(c2, "mask")
    m1 = sp.meta_prepare(i1, torch.bfloat16, M1, K1)
    m2 = sp.meta_prepare(i2, torch.bfloat16, M2, M1)
    X, Y0 = dev(c1["B"]), dev(c2["C"])
    Y1 = torch.empty((M1, N), dtype=torch.bfloat16, device="cuda")
    Y2 = torch.empty((M2, N), dtype=torch.float32, device="cuda")

    def poison():
        Y1.fill_(3.0e38)
        Y2.fill_(-3.0e38)

    def layers():
        sp.mma(v1, m1, X, None, out=Y1)
        sp.mma(v2, m2, Y1, Y0, out=Y2)

    if graph:
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                layers()
        torch.cuda.current_stream().wait_stream(side)
        for _ in range(2):
            poison()
            g.replay()
    else:
        poison()
        layers()
    torch.cuda.synchronize()
    assert int(s1.item()) == 0 and int(s2.item()) == 0
    # layer 1 against the oracle; layer 2 against the oracle applied to the Y1 the GPU made
    va, ia, _ = oracle.compress(inputs.bits(c1["A"]), "bf16", "mask", mask=c1["mask"].numpy())
    R1, S1 = oracle.mma_f64(va, ia, inputs.bits(c1["B"]), None, "bf16", "bf16", K1)
    check_float(Y1.float().cpu().numpy(), R1, S1, "bf16", "layer 1")
    vb, ib, _ = oracle.compress(inputs.bits(c2["A"]), "bf16", "mask", mask=c2["mask"].numpy())
    R2, S2 = oracle.mma_f64(vb, ib, inputs.bits(Y1.cpu()), inputs.bits(c2["C"]), "bf16", "bf16",
                            M1, tc="f32")
    check_float(Y2.cpu().numpy(), R2, S2, None, "layer 2")


@pytest.mark.parametrize("ta,tc,out,M,N,K", [
    ("bf16", "f32", torch.float32, 2500, 2296, 320),    # 90 tiles, ragged M, N and K
    ("f16", "bf16", torch.bfloat16, 3000, 2104, 288),  # 108 tiles, ragged M, N and K
])
def test_more_tiles_than_cta_pairs(ta, tc, out, M, N, K):
    # more 256 x 256 tiles than CTA pairs, with a last round that leaves pairs idle (its
    # tiles may run as halves): every element against the oracle
    c = inputs.case(ta, ta, M, N, K, seed=M + N, tc=tc)
    run_case(c, mode="mask", out_dtype=out)
