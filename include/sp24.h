/*
 * sp24.h -- C ABI of libsp24: 2:4 structured-sparse multiply-accumulate D = A_sp * B + C
 * on one GB300 (sm_103a).
 *
 * The operation is the one the sparse matrix-multiply builtins on these pages define:
 *   "RDNA4 sparse WMMA builtins", "Structured sparsity (2:4 pattern)": in every
 *     contiguous group of four elements of A along K exactly two are non-zero; A is
 *     stored as its packed non-zeros (half the K length) plus a sparsity index that
 *     gives, for each kept element, its 2-bit position 0-3 within the group;
 *   same page, "Builtin reference": every builtin returns
 *     expand(srcA, index) x srcB + srcC;
 *   "CDNA and CDNA2 sparse MFMA builtins", "Structured sparsity (4:2 pattern)" and the
 *     FP16 sparse kernels under "Using sparse MFMA builtins as a compute policy": the
 *     positions-0-and-2 pattern has the index byte 0x88 (two groups of four);
 *   "v_smfmac_f32_32x32x32_bf8_bf8", "Semantics": D = A (sparse) * B + D.
 *
 * Conventions for every entry point
 *   - All matrices are row-major; a leading dimension ("ld") counts elements (words for
 *     the index) between the starts of consecutive rows.
 *   - Pointers named d_* or documented as "device" are device pointers on the current
 *     CUDA device; `stream` is a cudaStream_t (NULL = legacy default stream).
 *   - The caller owns every buffer.  The library never allocates, frees or
 *     synchronises; all work is enqueued on `stream` and the call returns as soon as it
 *     is enqueued.
 *   - A synchronous return code reports argument and launch errors; nothing is enqueued
 *     when it is not SP24_OK.  Data-dependent conditions found on the device are OR-ed
 *     into the caller's 32-bit status word (nullable) as SP24_DEV_* bits; read it after
 *     the stream has synchronised.  The library never clears that word.
 *   - There is no CPU fallback: without an sm_103 device every compute call returns
 *     SP24_ERR_NO_DEVICE.
 *   - Stream order is kept as for any kernel, with one refinement: the products
 *     (sp24_mma*) are launched with programmatic stream serialisation, so a product
 *     may be placed on the GPU and run its set-up (shared-memory barriers, tensor-memory
 *     allocation) while the kernel before it on the stream is still running, and the next
 *     product on the stream may do the same while it runs.  A product reads or writes
 *     global memory only after the kernel before it has completed and its writes are
 *     visible, except that it may ask for the first part of its own A operand, metadata
 *     and B to be fetched into the L2 cache earlier (a hint with no effect on results).
 */
#ifndef SP24_H
#define SP24_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SP24_VERSION 1

/* Element types.  F16 = IEEE binary16, BF16 = bfloat16, E4M3 = OCP FP8 E4M3 (the
 * pages' "FP8"), E5M2 = OCP FP8 E5M2 (the pages' "BF8"), S8 / U8 = signed / unsigned
 * 8-bit integers (the a_neg / b_neg choice of "RDNA4 dense WMMA builtins", "Common
 * parameters"), F32 / S32 = accumulator and output types, S4 / U4 = signed (-8..7) /
 * unsigned (0..15) 4-bit integers ("RDNA4 sparse WMMA builtins", "INT4 and UINT4
 * inputs").  4-bit elements are stored two per byte, element 2i in the low nibble and
 * 2i+1 in the high nibble; their leading dimensions still count elements (a row pitch
 * of ld elements is ld/2 bytes). */
typedef enum sp24_dtype {
    SP24_F16 = 0,
    SP24_BF16 = 1,
    SP24_E4M3 = 2,
    SP24_E5M2 = 3,
    SP24_S8 = 4,
    SP24_U8 = 5,
    SP24_F32 = 6,
    SP24_S32 = 7,
    SP24_S4 = 8,
    SP24_U4 = 9
} sp24_dtype;

typedef enum sp24_status {
    SP24_OK = 0,
    SP24_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad K, ld too small   */
    SP24_ERR_UNSUPPORTED = 2, /* element-type combination not supported             */
    SP24_ERR_ALIGN = 3,       /* pointer or row pitch not 16-byte aligned           */
    SP24_ERR_CUDA = 4,        /* CUDA runtime or driver error while enqueueing      */
    SP24_ERR_TIMEOUT = 5,     /* reserved: the device reports timeouts via SP24_DEV_TIMEOUT */
    SP24_ERR_NOT_2_4 = 6,     /* reserved: the device reports this via SP24_DEV_NOT_2_4     */
    SP24_ERR_NO_DEVICE = 7,   /* no sm_103 device is current                        */
    SP24_ERR_SCRATCH_TOO_SMALL = 8 /* the problem needs more than the built-in scratch */
} sp24_status;

/* How sp24_compress chooses the two kept positions of each group of four. */
typedef enum sp24_mode {
    SP24_MODE_EXACT = 0,     /* the non-zero elements (the pages' host compression)  */
    SP24_MODE_MASK = 1,      /* the positions a byte mask marks (non-zero = keep)    */
    SP24_MODE_MAGNITUDE = 2  /* the two largest |x|; equal |x| -> the lower position */
} sp24_mode;

/* Device status bits, OR-ed into the caller's int32 status word. */
#define SP24_DEV_NOT_2_4 1 /* a group did not hold exactly two kept elements          */
#define SP24_DEV_TIMEOUT 2 /* a bounded wait inside a kernel gave up; output invalid  */

/*
 * sp24_compress -- dense (or masked) A -> packed values + sparsity index.
 *
 * Walks each row of A in groups of four along K and keeps two positions p0 < p1 per
 * group ("RDNA4 sparse WMMA builtins", "Structured sparsity (2:4 pattern)": extract the
 * two non-zero positions and pack them consecutively; the offline pruning pass of the
 * note under "Instantiating the kernel" is SP24_MODE_MAGNITUDE):
 *   values[i*ldv + 2g]   = A[i*lda + 4g + p0]      (bit copy)
 *   values[i*ldv + 2g+1] = A[i*lda + 4g + p1]
 *   index[i*ldi + g/8]   bits 4*(g%8) .. +3  = p0 | (p1 << 2)
 * (the nibble order is the one the CDNA example's literal 0x88 fixes for positions 0
 * and 2: the lower position in the low two bits).
 *
 * t      : SP24_F16, SP24_BF16, SP24_E4M3, SP24_E5M2, SP24_S8, SP24_U8, SP24_S4 or SP24_U4.
 * M, K   : rows and dense columns of A; K % 32 == 0 (one index word per 32 columns).
 * A      : device, M x K elements of type t, leading dimension lda >= K.
 * mask   : device, M x K bytes (ldm >= K), used only in SP24_MODE_MASK, else ignored.
 * values : device, M x K/2 elements of type t, ldv >= K/2.
 * index  : device, M x K/32 uint32 words, ldi >= K/32.
 * Group rules: EXACT keeps the non-zeros (+0 and -0 are zero); with fewer than two it
 * adds the lowest free positions, with more than two it keeps the two lowest and sets
 * SP24_DEV_NOT_2_4.  MASK keeps the marked positions by the same rules and sets
 * SP24_DEV_NOT_2_4 unless exactly two are marked.  MAGNITUDE never flags.
 * Alignment: A, values and mask 16-byte aligned; the row pitches of A and values (lda
 * and ldv elements of t) and ldm multiples of 16 bytes (for S4 / U4: lda and ldv
 * multiples of 32); index 4-byte aligned.  Otherwise SP24_ERR_ALIGN.
 */
sp24_status sp24_compress(sp24_dtype t, int64_t M, int64_t K, const void *A, int64_t lda,
                          const uint8_t *mask, int64_t ldm, sp24_mode mode, void *values,
                          int64_t ldv, uint32_t *index, int64_t ldi, int32_t *d_status,
                          void *stream);

/*
 * sp24_decompress -- the inverse: A[i][4g+p] = the kept value for p in {p0, p1}, zero
 * elsewhere (the expand() of "Builtin reference").  Same arguments, types and alignment
 * rules as sp24_compress; A is written.
 */
sp24_status sp24_decompress(sp24_dtype t, int64_t M, int64_t K, const void *values,
                            int64_t ldv, const uint32_t *index, int64_t ldi, void *A,
                            int64_t lda, void *stream);

/*
 * sp24_meta_bytes -- size in bytes of the metadata image sp24_meta_prepare writes for
 * an M x K (dense) operand of element type t; 0 for an unsupported t or bad size.
 */
size_t sp24_meta_bytes(sp24_dtype t, int64_t M, int64_t K);

/*
 * sp24_meta_prepare -- re-lay the canonical index (as sp24_compress writes it) into the
 * image from which sp24_mma fills tensor memory: for every 128-row tile of A and every K
 * step of the kernel (128 dense K for 16-bit types, 256 for FP8 types) one block of
 * 128 lanes x 16 bytes (16-bit types) or x 32 bytes (FP8 types), each lane holding its
 * words for the step's four MMAs.  Rows are padded to a multiple of 256 and K to the K
 * step; pad groups get the valid pattern {0,1} and their values are zero, so they add
 * nothing.  For whole tiles and steps the image is M x K / 8 bytes, the size of the
 * index.  It is a format private to sp24_mma (sp24_meta_bytes() gives its size); the
 * canonical index stays the interchange format.
 * 8- and 4-bit integer types use the layout of the 16-bit types (their product runs on
 * the bf16 tensor path).
 * index : device, M x K/32 words, ldi >= K/32, 4-byte aligned.
 * meta  : device, sp24_meta_bytes(t, M, K) bytes, 16-byte aligned.
 */
sp24_status sp24_meta_prepare(sp24_dtype t, int64_t M, int64_t K, const uint32_t *index,
                              int64_t ldi, void *meta, void *stream);

/*
 * sp24_compress_meta -- sp24_compress and sp24_meta_prepare in one pass over A: writes
 * values, the canonical index (optional) and the metadata image sp24_mma reads, with the
 * contents the two calls write.  One read of A instead of a read of A plus a read of the
 * index, and one launch instead of two ("Structured sparsity (2:4 pattern)": the
 * compression; the image is this library's own format for tensor memory).
 * Arguments as in sp24_compress, plus:
 * index : device or NULL (then no canonical index is written and ldi is ignored).
 * meta  : device, sp24_meta_bytes(t, M, K) bytes, 16-byte aligned.
 */
sp24_status sp24_compress_meta(sp24_dtype t, int64_t M, int64_t K, const void *A, int64_t lda,
                               const uint8_t *mask, int64_t ldm, sp24_mode mode, void *values,
                               int64_t ldv, uint32_t *index, int64_t ldi, void *meta,
                               int32_t *d_status, void *stream);

/*
 * sp24_mma_workspace_bytes -- device workspace sp24_mma needs for (ta, tb, M, N, K): for
 * integer operands the bytes of both operands widened to bf16 (A_c: M x K/2, B: K x N
 * with the row pitch rounded up to 8 elements); 0 for float operands.
 */
size_t sp24_mma_workspace_bytes(sp24_dtype ta, sp24_dtype tb, int64_t M, int64_t N, int64_t K);

/*
 * sp24_mma -- D = expand(values, index) * B + C, the sparse product of "Builtin reference"
 * (expand(srcA, index) x srcB + srcC) on the tcgen05 sparse tensor cores.
 *
 * ta, tb, tc, td supported combinations (anything else: SP24_ERR_UNSUPPORTED):
 *   (F16, F16) and (BF16, BF16)     -> f32 accumulate, tc in {F32, F16, BF16, none},
 *                                      td in {F32, F16, BF16}
 *   (E4M3, E4M3), (E5M2, E5M2),
 *   (E4M3, E5M2) and (E5M2, E4M3)   -> the same C and D types
 *   (S8, S8) and (U8, S8)           -> exact integer result, tc in {S32, none}, td = S32,
 *                                      32-bit two's-complement wrap, no clamp
 *   (S4 or U4, S4 or U4)            -> the same, for 4-bit operands (any sign mix)
 * "none" for tc means C == NULL (treated as zero); tc is then ignored.
 * M, N, K : D is M x N; K is the dense depth, K % 32 == 0.
 * values  : device, M x K/2 of ta (ldv >= K/2), from sp24_compress.
 * meta    : device, the image sp24_meta_prepare wrote for (ta, M, K).
 * B       : device, K x N of tb, row-major (ldb >= N).
 * C       : device or NULL, M x N of tc (ldc >= N).      D : device, M x N of td (ldd >= N).
 * workspace, workspace_bytes : device scratch of at least sp24_mma_workspace_bytes(),
 *           16-byte aligned, owned by the caller and used only by this call's kernels
 *           (integer operands only; NULL / 0 otherwise).
 * Leading dimensions count elements, also for 4-bit types (two per byte).
 * Accumulation: floats in f32 on the tensor cores; a 16-bit C is widened exactly and a
 * BF16 or F16 D is the f32 result rounded to nearest-even once.  (F16, F16, F16, F16) and
 * (BF16, BF16, BF16, BF16) are the FP16- / BF16-accumulate forms of "RDNA4 sparse WMMA
 * builtins"; summing in f32 and rounding once is at least as accurate as 16-bit sums.
 * Integers are widened to bf16 (exact) and accumulated in f32 in chunks whose sums are
 * exact integers of at most 2^24 (2048 dense K for S8 x S8, 1024 for U8 x S8, 8192 for
 * 4-bit operands), the chunks then summed in int32: the result is exact.  (A u8 x u8
 * chunk of even 1024 K could pass 2^24, hence B = S8 for 8-bit operands.)
 * Alignment: values, meta, B, C, D 16-byte aligned, every row pitch a multiple of 16 bytes.
 * Device status: SP24_DEV_TIMEOUT if a pipeline wait gave up (D is then invalid).
 */
sp24_status sp24_mma(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td,
                     int64_t M, int64_t N, int64_t K, const void *values, int64_t ldv,
                     const void *meta, const void *B, int64_t ldb, const void *C,
                     int64_t ldc, void *D, int64_t ldd, void *workspace,
                     size_t workspace_bytes, int32_t *d_status, void *stream);

/*
 * sp24_mma_index -- sp24_mma with the sparsity metadata read from the canonical index
 * itself (as sp24_compress writes it: M x K/32 words, group g of row i in bits
 * 4(g%8)..+3 of word g/8, nibble = p0 | p1 << 2, "Structured sparsity (2:4 pattern)")
 * instead of the image: no sp24_meta_prepare pass and no image buffer.  The kernel's
 * writer warps permute the words into tensor memory themselves.  Results are bit-identical
 * to sp24_mma on sp24_meta_prepare(index).
 * index : device, M x K/32 words, ldi >= K/32, 4-byte aligned (any pitch).
 * Every other argument, type combination and rule as in sp24_mma.
 */
sp24_status sp24_mma_index(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td,
                           int64_t M, int64_t N, int64_t K, const void *values, int64_t ldv,
                           const uint32_t *index, int64_t ldi, const void *B, int64_t ldb,
                           const void *C, int64_t ldc, void *D, int64_t ldd, void *workspace,
                           size_t workspace_bytes, int32_t *d_status, void *stream);

/*
 * sp24_diag_wait_timeout -- self-test of the bounded waits every kernel uses.  Launches
 * one thread that waits on a barrier nothing ever arrives at; after limit_ns nanoseconds
 * the wait gives up and SP24_DEV_TIMEOUT is OR-ed into *d_status (device, 4 bytes).  The
 * context stays usable.  It exists so that the give-up path can be tested without a
 * faulting or hanging GPU.
 */
sp24_status sp24_diag_wait_timeout(int32_t *d_status, uint64_t limit_ns, void *stream);

/*
 * sp24_diag_mma_stall -- self-test of the sparse product's give-up path.  Launches the very
 * kernel sp24_mma runs for a float problem of this shape (ta = tb = f16, bf16, E4M3 or
 * E5M2; no C; f32 D), except that its TMA producer issues no copies, so the operands of the
 * first stage never arrive.  Every wait of the kernel is bounded by limit_ns nanoseconds
 * (0 < limit_ns <= 1 s): the MMA thread's wait gives up, the other roles see that (or give
 * up themselves), the CTAs let their metadata stores finish, free their tensor memory and
 * exit, and SP24_DEV_TIMEOUT is OR-ed into *d_status.  values / meta / B / D must be valid
 * device buffers as for sp24_mma (the metadata writers read the first stages' words of
 * meta); D is left unwritten.  No copy or MMA is in flight when the kernel exits, so the
 * context stays usable.  The source pages have no counterpart: it exists so that the
 * failure path is exercised without faulting or hanging a GPU.
 */
sp24_status sp24_diag_mma_stall(sp24_dtype ta, int64_t M, int64_t N, int64_t K,
                                const void *values, int64_t ldv, const void *meta, const void *B,
                                int64_t ldb, void *D, int64_t ldd, uint64_t limit_ns,
                                int32_t *d_status, void *stream);

/* Bytes of the fixed device scratch array sp24_mma_i8_noalloc uses (16 MiB). */
#define SP24_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * sp24_mma_strided_batched -- `batch` independent products of one shape in one launch
 * (e.g. the same layer for several sequences, or experts of equal size):
 *   D_b = expand(values_b, meta_b) * B_b + C_b,  b = 0 .. batch-1,
 * where operand X of problem b starts at X + b * stride_X.  The tiles of all problems
 * are scheduled together, so small problems fill the GPU.  Float operands only (the
 * pairs sp24_mma takes for 16-bit and FP8 types); everything else as in sp24_mma for each
 * problem (sizes, leading dimensions, alignment, tc / td, status bits).
 * stride_values, stride_b : elements of ta / tb between problems' values and B.
 * stride_meta : bytes between problems' metadata images, >= sp24_meta_bytes(ta, M, K).
 * stride_c, stride_d : elements between problems' C and D; D blocks must not overlap
 *   (stride_d >= M * ldd).  Every stride times its element size is a multiple of 16 bytes.
 * batch == 0: nothing is enqueued; batch == 1 is sp24_mma without a workspace.
 */
sp24_status sp24_mma_strided_batched(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc,
                                     sp24_dtype td, int64_t batch, int64_t M, int64_t N,
                                     int64_t K, const void *values, int64_t ldv,
                                     int64_t stride_values, const void *meta,
                                     int64_t stride_meta, const void *B, int64_t ldb,
                                     int64_t stride_b, const void *C, int64_t ldc,
                                     int64_t stride_c, void *D, int64_t ldd, int64_t stride_d,
                                     int32_t *d_status, void *stream);

/* One problem of a grouped product (all fields as the sp24_mma arguments of that name). */
typedef struct sp24_mma_problem {
    int64_t M, N, K;
    const void *values; int64_t ldv;
    const void *meta;
    const void *B; int64_t ldb;
    const void *C; int64_t ldc;   /* C may be NULL */
    void *D; int64_t ldd;
} sp24_mma_problem;

/*
 * sp24_mma_grouped -- D_g = expand(values_g, meta_g) * B_g + C_g for `count` problems of
 * different shapes (e.g. the experts of a mixture-of-experts layer with their own token
 * counts), one persistent launch per 32 problems whose tiles share the GPU.  Float
 * operands only, one (ta, tb, tc, td) combination for all problems (the pairs and C / D
 * types sp24_mma takes for 16-bit and FP8 operands); every problem is validated as
 * sp24_mma validates its arguments, and nothing is enqueued if any problem fails.
 * Problems with M == 0 or N == 0 are skipped.  The tile shape follows the widest N of
 * each launch's problems.  problems: host array, read during the call only.
 */
sp24_status sp24_mma_grouped(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td,
                             const sp24_mma_problem *problems, int64_t count,
                             int32_t *d_status, void *stream);

/*
 * sp24_mma_i8_noalloc -- the 8-bit integer form of sp24_mma without a workspace argument.
 * The source pages have no counterpart; this entry point exists for callers that cannot
 * allocate device memory at the point of the call: for example a plugin inside a host
 * framework that owns all device memory and hands out no workspace, or a caller with a
 * fixed memory plan that forbids allocations after start-up (cudaMalloc may also
 * synchronise the device).  It allocates nothing and calls no allocating routine.
 *
 * Arguments, types and results are those of sp24_mma for (S8, S8) and (U8, S8) operands
 * (tc in {S32, none}, td = S32).  The scratch for the operands widened to bf16 is a device
 * array of SP24_NOALLOC_SCRATCH_BYTES inside the library, held by every GPU that loads it
 * until the process exits; a problem needing more than that (sp24_mma_workspace_bytes())
 * returns SP24_ERR_SCRATCH_TOO_SMALL and enqueues nothing.  All calls share the array and
 * each call writes what it uses before reading it; calls whose work overlaps on the GPU
 * (no stream ordering between them) race on it.  The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current); make that first
 * call before any stream capture.  The address is kept per device and context: after the
 * context is destroyed (cudaDeviceReset) the array's contents are gone, and the next call
 * in the new context looks the address up again.
 */
sp24_status sp24_mma_i8_noalloc(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td,
                                int64_t M, int64_t N, int64_t K, const void *values,
                                int64_t ldv, const void *meta, const void *B, int64_t ldb,
                                const void *C, int64_t ldc, void *D, int64_t ldd,
                                int32_t *d_status, void *stream);

/* Static description of a status code (never NULL). */
const char *sp24_status_string(sp24_status s);

/* SP24_VERSION of the loaded library. */
int sp24_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SP24_H */
