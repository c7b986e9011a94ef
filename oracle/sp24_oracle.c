/*
 * sp24_oracle.c -- plain CPU oracle for the 2:4 structured-sparse multiply-accumulate.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE: only the test suite, the smoke check in
 * __graft_entry__.py and the CPU-baseline / reference legs of bench.py use it.  It is
 * deliberately slow and literal: no blocking, no fusion, double (or int64) arithmetic,
 * one element at a time.  See sp24_oracle.h for the page citations.
 */
#include "sp24_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int or_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int or_elem_bytes(int dtype)
{
    switch (dtype) {
    case OR_F16:
    case OR_BF16:
        return 2;
    case OR_E4M3:
    case OR_E5M2:
    case OR_S8:
    case OR_U8:
    case OR_S4: /* one element per byte in the oracle's arrays */
    case OR_U4:
        return 1;
    case OR_F32:
    case OR_S32:
        return 4;
    default:
        return 0;
    }
}

/* ---------------------------------------------------------------------------------
 * Element decoding, each written out from its format definition (sign, biased
 * exponent, fraction; exponent 0 = subnormal).  The FP8 pair is the OCP definition:
 * E4M3 has bias 7, no infinities, and only S.1111.111 is NaN (max 448); E5M2 has bias
 * 15 and IEEE-style inf/NaN (max 57344).  The pages name these formats "FP8 (E4M3)"
 * and "BF8 (E5M2)" ("RDNA4 sparse WMMA builtins", "FP8 and BF8 inputs").
 * --------------------------------------------------------------------------------- */
static double dec_float(uint32_t bits, int ebits, int mbits, int bias, int ieee_special)
{
    uint32_t s = (bits >> (ebits + mbits)) & 1u;
    uint32_t e = (bits >> mbits) & ((1u << ebits) - 1u);
    uint32_t m = bits & ((1u << mbits) - 1u);
    uint32_t emax = (1u << ebits) - 1u;
    double v;
    if (e == 0) {
        /* subnormal: 0.m * 2^(1-bias) = m * 2^(1-bias-mbits) */
        v = ldexp((double)m, 1 - bias - mbits);
    } else if (e == emax && ieee_special) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        /* normal: 1.m * 2^(e-bias) = (2^mbits + m) * 2^(e-bias-mbits) */
        v = ldexp((double)((1u << mbits) + m), (int)e - bias - mbits);
    }
    return s ? -v : v;
}

double or_decode(int dtype, uint32_t bits)
{
    switch (dtype) {
    case OR_F16:
        return dec_float(bits & 0xffffu, 5, 10, 15, 1);
    case OR_BF16:
        return dec_float(bits & 0xffffu, 8, 7, 127, 1);
    case OR_E4M3:
        /* no infinities; exponent 15 is an ordinary binade except mantissa 7 = NaN */
        if ((bits & 0x7fu) == 0x7fu)
            return NAN;
        return dec_float(bits & 0xffu, 4, 3, 7, 0);
    case OR_E5M2:
        return dec_float(bits & 0xffu, 5, 2, 15, 1);
    case OR_S8:
        return (double)(int8_t)(uint8_t)bits;
    case OR_U8:
        return (double)(uint8_t)bits;
    case OR_S4: /* 4-bit two's complement: -8 .. 7 ("iu4" with the sign flag set) */
        return (double)((int)(bits & 0xfu) - (int)((bits & 0x8u) << 1));
    case OR_U4:
        return (double)(bits & 0xfu);
    case OR_F32:
        return dec_float(bits, 8, 23, 127, 1);
    case OR_S32:
        return (double)(int32_t)bits;
    default:
        return NAN;
    }
}

uint16_t or_round_bf16(double x)
{
    if (isnan(x))
        return 0x7fc0u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double ax = fabs(x);
    if (ax == 0.0)
        return sign;
    /* quantum of the bf16 binade holding ax: 8 significant bits, min exponent -126 */
    int e;
    frexp(ax, &e); /* ax = f * 2^e, f in [0.5, 1): unbiased exponent is e-1 */
    int ue = e - 1;
    if (ue < -126)
        ue = -126; /* subnormal range has the fixed quantum 2^-133 */
    double q = ldexp(1.0, ue - 7);
    double y = rint(ax / q) * q; /* ax/q is exact; rint rounds half to even */
    if (y >= ldexp(1.0, 128))
        return sign | 0x7f80u; /* overflow to infinity */
    /* y now holds at most 8 significant bits: it is exact in binary32, whose upper
     * half is the bfloat16 pattern. */
    float f = (float)y;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

uint16_t or_round_f16(double x)
{
    if (isnan(x))
        return 0x7e00u;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double ax = fabs(x);
    if (ax == 0.0)
        return sign;
    /* quantum of the binary16 binade holding ax: 11 significant bits, min exponent -14 */
    int e;
    frexp(ax, &e);
    int ue = e - 1;
    if (ue < -14)
        ue = -14; /* subnormal range has the fixed quantum 2^-24 */
    double q = ldexp(1.0, ue - 10);
    double y = rint(ax / q) * q; /* ties to even */
    if (y >= 65536.0)
        return sign | 0x7c00u; /* overflow to infinity (65520 and above) */
    if (y < ldexp(1.0, -14))   /* subnormal (or the smallest normal reached by rounding) */
        return (uint16_t)(sign | (uint16_t)(y / ldexp(1.0, -24)));
    frexp(y, &e);
    ue = e - 1;
    uint32_t frac = (uint32_t)(y / ldexp(1.0, ue - 10)) - 1024u; /* 10 fraction bits */
    return (uint16_t)(sign | (uint16_t)((uint32_t)(ue + 15) << 10) | (uint16_t)frac);
}

int32_t or_wrap_i32(int64_t x)
{
    uint32_t u = (uint32_t)((uint64_t)x & 0xffffffffu);
    int32_t r;
    memcpy(&r, &u, 4);
    return r;
}

static uint32_t load_bits(const void *base, int esz, int64_t off);

void or_decode_array(int dtype, const void *src, int64_t n, double *dst)
{
    int esz = or_elem_bytes(dtype);
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_decode(dtype, load_bits(src, esz, i));
}

void or_round_bf16_array(const double *src, int64_t n, uint16_t *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_round_bf16(src[i]);
}

void or_round_f16_array(const double *src, int64_t n, uint16_t *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_round_f16(src[i]);
}

void or_wrap_i32_array(const int64_t *src, int64_t n, int32_t *dst)
{
    for (int64_t i = 0; i < n; ++i)
        dst[i] = or_wrap_i32(src[i]);
}

static uint32_t load_bits(const void *base, int esz, int64_t off)
{
    const uint8_t *p = (const uint8_t *)base + off * esz;
    uint32_t v = 0;
    memcpy(&v, p, (size_t)esz); /* little-endian element */
    return v;
}

static void store_bits(void *base, int esz, int64_t off, uint32_t v)
{
    memcpy((uint8_t *)base + off * esz, &v, (size_t)esz);
}

/* ---------------------------------------------------------------------------------
 * Compression: "walk the K dimension in groups of four, extract the two non-zero
 * positions, and pack them consecutively" ("RDNA4 sparse WMMA builtins" and "CDNA and
 * CDNA2 sparse MFMA builtins", structured-sparsity sections).  The index holds, per
 * group, the two 2-bit positions ("Common parameters": each pair of bits is the
 * position 0-3 of one non-zero in its block of four).  The CDNA example passes 0x88
 * for the positions-0-and-2 pattern on two groups, i.e. a nibble 0b10'00: the lower
 * position in the low two bits.  Groups are packed eight per 32-bit word, group g at
 * bit 4*(g mod 8) of word g/8.
 *
 * Readings where the pages are silent:
 *   exact mode, fewer than two non-zeros: fill with the lowest unused positions;
 *   exact mode, more than two non-zeros:  keep the two lowest, flag the group;
 *   mask mode, count != 2:                same fill / keep-lowest rule, flag the group;
 *   magnitude mode: rank by (|x| descending, position ascending), keep the top two.
 * --------------------------------------------------------------------------------- */
int64_t or_compress(int dtype, int64_t M, int64_t K, const void *A, int64_t lda,
                    const uint8_t *mask, int64_t ldm, int mode, void *values,
                    int64_t ldv, uint32_t *index, int64_t ldi, uint8_t *flags)
{
    int esz = or_elem_bytes(dtype);
    if (esz == 0 || esz == 4 || (K % 4) != 0 || (mode == OR_MODE_MASK && !mask))
        return -1;
    int64_t groups = K / 4;
    int64_t words = (groups + 7) / 8;
    int64_t nflag = 0;

    for (int64_t i = 0; i < M; ++i) {
        for (int64_t w = 0; w < words; ++w)
            index[i * ldi + w] = 0u;
        for (int64_t g = 0; g < groups; ++g) {
            uint32_t x[4];
            double d[4];
            int sel[4];
            int nsel = 0;
            for (int p = 0; p < 4; ++p) {
                x[p] = load_bits(A, esz, i * lda + 4 * g + p);
                d[p] = or_decode(dtype, x[p]);
            }
            int p0 = -1, p1 = -1, flagged = 0;
            if (mode == OR_MODE_MAGNITUDE) {
                /* largest |x| first; on equal |x| the lower position wins */
                int best = 0;
                for (int p = 1; p < 4; ++p)
                    if (fabs(d[p]) > fabs(d[best]))
                        best = p;
                int second = (best == 0) ? 1 : 0;
                for (int p = 0; p < 4; ++p)
                    if (p != best && fabs(d[p]) > fabs(d[second]))
                        second = p;
                p0 = best < second ? best : second;
                p1 = best < second ? second : best;
            } else {
                for (int p = 0; p < 4; ++p) {
                    int keep = (mode == OR_MODE_MASK) ? (mask[i * ldm + 4 * g + p] != 0)
                                                      : (d[p] != 0.0 || isnan(d[p]));
                    if (keep)
                        sel[nsel++] = p;
                }
                if (mode == OR_MODE_MASK ? (nsel != 2) : (nsel > 2))
                    flagged = 1;
                /* fill up to two with the lowest positions not yet chosen */
                for (int p = 0; p < 4 && nsel < 2; ++p) {
                    int used = 0;
                    for (int s = 0; s < nsel; ++s)
                        used |= (sel[s] == p);
                    if (!used) {
                        sel[nsel++] = p;
                    }
                }
                /* Without a fill sel is ascending, so sel[0], sel[1] are the two lowest
                 * chosen positions; after a fill the pair may be out of order. */
                int a = sel[0], b = sel[1];
                p0 = a < b ? a : b;
                p1 = a < b ? b : a;
            }
            store_bits(values, esz, i * ldv + 2 * g, x[p0]);
            store_bits(values, esz, i * ldv + 2 * g + 1, x[p1]);
            uint32_t nib = (uint32_t)p0 | ((uint32_t)p1 << 2);
            index[i * ldi + g / 8] |= nib << (4 * (g % 8));
            if (flags)
                flags[i * groups + g] = flagged ? OR_FLAG_NOT_2_4 : 0;
            nflag += flagged;
        }
    }
    return nflag;
}

/* expand(srcA, index): the kept values go back to positions 4g+p0 and 4g+p1 of their
 * group; the two other positions of the group are zero. */
void or_decompress(int dtype, int64_t M, int64_t K, const void *values, int64_t ldv,
                   const uint32_t *index, int64_t ldi, void *A, int64_t lda)
{
    int esz = or_elem_bytes(dtype);
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t k = 0; k < K; ++k)
            store_bits(A, esz, i * lda + k, 0u);
        for (int64_t g = 0; g < K / 4; ++g) {
            uint32_t nib = (index[i * ldi + g / 8] >> (4 * (g % 8))) & 0xfu;
            int p0 = (int)(nib & 3u), p1 = (int)(nib >> 2);
            store_bits(A, esz, i * lda + 4 * g + p0, load_bits(values, esz, i * ldv + 2 * g));
            store_bits(A, esz, i * lda + 4 * g + p1,
                       load_bits(values, esz, i * ldv + 2 * g + 1));
        }
    }
}

/* one decoded row of expand(values, index), dense length K */
static void expand_row_f64(int ta, int64_t K, const void *values, int64_t ldv,
                           const uint32_t *index, int64_t ldi, int64_t i, double *row)
{
    int esz = or_elem_bytes(ta);
    for (int64_t k = 0; k < K; ++k)
        row[k] = 0.0;
    for (int64_t g = 0; g < K / 4; ++g) {
        uint32_t nib = (index[i * ldi + g / 8] >> (4 * (g % 8))) & 0xfu;
        int p0 = (int)(nib & 3u), p1 = (int)(nib >> 2);
        row[4 * g + p0] = or_decode(ta, load_bits(values, esz, i * ldv + 2 * g));
        row[4 * g + p1] = or_decode(ta, load_bits(values, esz, i * ldv + 2 * g + 1));
    }
}

static int valid_ab(int t) { return t >= OR_F16 && t <= OR_U8; }

/* D = expand(A, index) * B + C ("Builtin reference": expand(srcA, index) x srcB + srcC;
 * "v_smfmac_f32_32x32x32_bf8_bf8" Semantics: D = A(sparse) * B + D), in double.  The
 * loop order is i-k-j; a zero a_ik adds nothing and is skipped.  C may be f32, s32, or
 * the 16-bit accumulators of "FP16-accumulate builtins" / "BF16-accumulate builtins". */
int or_mma_f64(int ta, int tb, int64_t M, int64_t N, int64_t K, const void *values,
               int64_t ldv, const uint32_t *index, int64_t ldi, const void *B,
               int64_t ldb, int tc, const void *C, int64_t ldc, const int64_t *rows,
               int64_t nrows, double *D, double *S)
{
    if (!valid_ab(ta) || !valid_ab(tb) ||
        (C && tc != OR_F32 && tc != OR_S32 && tc != OR_F16 && tc != OR_BF16))
        return -1;
    (void)M;
    int besz = or_elem_bytes(tb);
    int cesz = C ? or_elem_bytes(tc) : 0;
    /* decode table for B's element type, built from or_decode */
    int nlut = (besz == 2) ? 65536 : 256;
    double *lut = (double *)malloc(sizeof(double) * (size_t)nlut);
    if (!lut)
        return -2;
    for (int v = 0; v < nlut; ++v)
        lut[v] = or_decode(tb, (uint32_t)v);

#pragma omp parallel
    {
        double *arow = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t i = rows ? rows[r] : r;
            double *drow = D + r * N;
            double *srow = S + r * N;
            for (int64_t j = 0; j < N; ++j) {
                drow[j] = C ? or_decode(tc, load_bits(C, cesz, i * ldc + j)) : 0.0;
                srow[j] = 0.0;
            }
            expand_row_f64(ta, K, values, ldv, index, ldi, i, arow);
            for (int64_t k = 0; k < K; ++k) {
                double a = arow[k];
                if (a == 0.0)
                    continue;
                for (int64_t j = 0; j < N; ++j) {
                    double p = a * lut[load_bits(B, besz, k * ldb + j)];
                    drow[j] += p;
                    srow[j] += fabs(p);
                }
            }
        }
        free(arow);
    }
    free(lut);
    return 0;
}

static int is_int_ab(int t) { return t == OR_S8 || t == OR_U8 || t == OR_S4 || t == OR_U4; }

/* Integer form: 8- or 4-bit operands (a_neg / b_neg pick signed or unsigned, "Common
 * parameters"; 4-bit is the pages' iu4), exact int64 sums, C of type s32 or absent. */
int or_mma_i64(int ta, int tb, int64_t M, int64_t N, int64_t K, const void *values,
               int64_t ldv, const uint32_t *index, int64_t ldi, const void *B,
               int64_t ldb, const void *C, int64_t ldc, const int64_t *rows,
               int64_t nrows, int64_t *D)
{
    if (!is_int_ab(ta) || !is_int_ab(tb))
        return -1;
    (void)M;
#pragma omp parallel
    {
        int64_t *arow = (int64_t *)malloc(sizeof(int64_t) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            int64_t i = rows ? rows[r] : r;
            int64_t *drow = D + r * N;
            for (int64_t j = 0; j < N; ++j)
                drow[j] = C ? (int64_t)(int32_t)load_bits(C, 4, i * ldc + j) : 0;
            for (int64_t k = 0; k < K; ++k)
                arow[k] = 0;
            for (int64_t g = 0; g < K / 4; ++g) {
                uint32_t nib = (index[i * ldi + g / 8] >> (4 * (g % 8))) & 0xfu;
                int p0 = (int)(nib & 3u), p1 = (int)(nib >> 2);
                uint32_t v0 = load_bits(values, 1, i * ldv + 2 * g);
                uint32_t v1 = load_bits(values, 1, i * ldv + 2 * g + 1);
                arow[4 * g + p0] = (int64_t)or_decode(ta, v0);
                arow[4 * g + p1] = (int64_t)or_decode(ta, v1);
            }
            for (int64_t k = 0; k < K; ++k) {
                int64_t a = arow[k];
                if (a == 0)
                    continue;
                const uint8_t *brow = (const uint8_t *)B + k * ldb;
                for (int64_t j = 0; j < N; ++j) {
                    int64_t b = (int64_t)or_decode(tb, brow[j]);
                    drow[j] += a * b;
                }
            }
        }
        free(arow);
    }
    return 0;
}
