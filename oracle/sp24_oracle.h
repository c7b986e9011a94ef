/*
 * sp24_oracle.h -- plain CPU oracle for the 2:4 structured-sparse multiply-accumulate.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check in
 * __graft_entry__.py and the CPU-baseline / reference legs of bench.py may load or call
 * this library.  It shares no code, header, table or helper with the CUDA library; the
 * type and mode codes below are this file's own and are mapped by name in the Python
 * wrapper.
 *
 * Every function is written from the definitions on these pages:
 *   [RDNA4-SP]  "RDNA4 sparse WMMA builtins": "Structured sparsity (2:4 pattern)",
 *               "Common parameters", "Builtin reference" (every builtin returns
 *               expand(srcA, index) x srcB + srcC).
 *   [CDNA-SP]   "CDNA and CDNA2 sparse MFMA builtins": "Structured sparsity (4:2 pattern)",
 *               "Using sparse MFMA builtins as a compute policy" (index literal 0x88 for
 *               the positions-0-and-2 pattern).
 *   [RDNA4-WM]  "RDNA4 dense WMMA builtins": "Common parameters" (a_neg / b_neg choose
 *               signed or unsigned integer operands).
 *   [CDNA4-ISA] "v_smfmac_f32_32x32x32_bf8_bf8": "Semantics" (D = A_sparse * B + D).
 */
#ifndef SP24_ORACLE_H
#define SP24_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types (this oracle's own numbering) */
enum {
    OR_F16 = 0,   /* IEEE binary16                                       */
    OR_BF16 = 1,  /* bfloat16: the upper half of an IEEE binary32        */
    OR_E4M3 = 2,  /* OCP FP8 E4M3 (finite only, max 448): the pages' FP8 */
    OR_E5M2 = 3,  /* OCP FP8 E5M2 (max 57344): the pages' BF8            */
    OR_S8 = 4,    /* signed 8-bit integer   (a_neg / b_neg = true)       */
    OR_U8 = 5,    /* unsigned 8-bit integer (a_neg / b_neg = false)      */
    OR_F32 = 6,   /* IEEE binary32 (C operand only)                      */
    OR_S32 = 7,   /* 32-bit two's complement (C operand only)            */
    OR_S4 = 8,    /* signed 4-bit integer (the pages' iu4 with a_neg / b_neg set),
                     one element per byte here, pattern in the low nibble */
    OR_U4 = 9     /* unsigned 4-bit integer, stored like OR_S4            */
};

/* compression modes */
enum {
    OR_MODE_EXACT = 0,     /* keep the non-zeros of each group of four          */
    OR_MODE_MASK = 1,      /* keep the positions a caller-supplied mask marks   */
    OR_MODE_MAGNITUDE = 2  /* keep the two largest |x| per group, ties -> lower */
};

/* per-group flag written by or_compress */
#define OR_FLAG_NOT_2_4 1

int or_elem_bytes(int dtype);

/* Exact value of one stored element (bit pattern in the low bits of `bits`). */
double or_decode(int dtype, uint32_t bits);

/* Round a real number to the nearest bfloat16, ties to even; returns the bit pattern. */
uint16_t or_round_bf16(double x);

/* Round a real number to the nearest IEEE binary16, ties to even (65520 and above ->
 * infinity); returns the bit pattern.  The FP16-accumulate result of "RDNA4 sparse WMMA
 * builtins" is read as the exact sum rounded once to this format. */
uint16_t or_round_f16(double x);

/* Two's-complement wrap of an exact integer sum to 32 bits. */
int32_t or_wrap_i32(int64_t x);

/* Array forms of the three functions above (n elements each). */
void or_decode_array(int dtype, const void *src, int64_t n, double *dst);
void or_round_bf16_array(const double *src, int64_t n, uint16_t *dst);
void or_round_f16_array(const double *src, int64_t n, uint16_t *dst);
void or_wrap_i32_array(const int64_t *src, int64_t n, int32_t *dst);

/*
 * Compress a dense M x K matrix A (row-major, leading dimension lda elements) whose rows
 * are split into groups of four along K.  For group g of row i the two kept positions
 * p0 < p1 are chosen by `mode`; values[i*ldv + 2g] = A[i][4g+p0],
 * values[i*ldv + 2g+1] = A[i][4g+p1] (bit copies), and the nibble (p0 | p1 << 2) is
 * stored at bits 4*(g%8) of index[i*ldi + g/8].  mask (MODE_MASK only) is M x K bytes
 * with leading dimension ldm, non-zero = keep.  K must be a multiple of 4; the unused
 * high nibbles of a row's last word (K % 32 != 0) are written as zero.
 * Returns the number of groups that broke the 2:4 rule (flagged groups);
 * flags (nullable, M x K/4 bytes) receives OR_FLAG_NOT_2_4 per flagged group.
 */
int64_t or_compress(int dtype, int64_t M, int64_t K, const void *A, int64_t lda,
                    const uint8_t *mask, int64_t ldm, int mode, void *values,
                    int64_t ldv, uint32_t *index, int64_t ldi, uint8_t *flags);

/* Inverse of compression: scatter the kept values back, every other position zero. */
void or_decompress(int dtype, int64_t M, int64_t K, const void *values, int64_t ldv,
                   const uint32_t *index, int64_t ldi, void *A, int64_t lda);

/*
 * D = expand(values, index) * B + C for the rows listed in rows[0..nrows) (all rows
 * 0..M-1 when rows == NULL, nrows == M), accumulated in double from the exact decoded
 * inputs.  B is K x N row-major (ldb), C (nullable => 0) is M x N (ldc) of type tc
 * (OR_F32 or OR_S32).  D and S are nrows x N, row-major; S receives sum_k |a_ik * b_kj|
 * (the scale of the tolerance).  Returns 0, or -1 on a bad type code.
 */
int or_mma_f64(int ta, int tb, int64_t M, int64_t N, int64_t K, const void *values,
               int64_t ldv, const uint32_t *index, int64_t ldi, const void *B,
               int64_t ldb, int tc, const void *C, int64_t ldc, const int64_t *rows,
               int64_t nrows, double *D, double *S);

/* Integer variant: exact int64 sums for S8/U8/S4/U4 operands (C of type OR_S32 or NULL). */
int or_mma_i64(int ta, int tb, int64_t M, int64_t N, int64_t K, const void *values,
               int64_t ldv, const uint32_t *index, int64_t ldi, const void *B,
               int64_t ldb, const void *C, int64_t ldc, const int64_t *rows,
               int64_t nrows, int64_t *D);

/* Number of OpenMP threads the product routines use (1 without OpenMP). */
int or_num_threads(void);

#ifdef __cplusplus
}
#endif
#endif
