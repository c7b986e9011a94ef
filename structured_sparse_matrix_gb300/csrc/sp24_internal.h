// sp24_internal.h -- host-side declarations shared by the translation units of libsp24.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

struct sp24_mma_problem;  // include/sp24.h

namespace sp24 {

// element codes: identical to sp24_dtype in include/sp24.h
enum : int {
  kF16 = 0, kBF16 = 1, kE4M3 = 2, kE5M2 = 3, kS8 = 4, kU8 = 5, kF32 = 6, kS32 = 7,
  kS4 = 8, kU4 = 9
};

// bits per element (4-bit types: two per byte, element 2i in the low nibble)
inline int elem_bits(int t) {
  switch (t) {
    case kF16: case kBF16: return 16;
    case kE4M3: case kE5M2: case kS8: case kU8: return 8;
    case kF32: case kS32: return 32;
    case kS4: case kU4: return 4;
    default: return 0;
  }
}
// bytes of a whole-byte type (0 for 4-bit types)
inline int dtype_bytes(int t) { return elem_bits(t) >= 8 ? elem_bits(t) / 8 : 0; }
// row pitch in bytes of `ld` elements; ld_ok16: that pitch is a whole number of 16-byte
// units (for 4-bit types this also makes ld even)
inline int64_t ld_bytes(int t, int64_t ld) { return ld * elem_bits(t) / 8; }
inline bool ld_ok16(int t, int64_t ld) { return (ld * elem_bits(t)) % 128 == 0; }
inline bool is_ab_type(int t) { return (t >= kF16 && t <= kU8) || t == kS4 || t == kU4; }
inline bool is_f8(int t) { return t == kE4M3 || t == kE5M2; }
inline bool is_i8(int t) { return t == kS8 || t == kU8; }
inline bool is_i4(int t) { return t == kS4 || t == kU4; }
inline bool is_int(int t) { return is_i8(t) || is_i4(t); }
inline bool is_signed_int(int t) { return t == kS8 || t == kS4; }
// C and D types of the float products: f32, or the 16-bit accumulators
inline bool is_float_acc(int t) { return t == kF32 || t == kBF16 || t == kF16; }

// ---- sparse-GEMM K-step geometry (one pipeline stage) shared by meta.cu, compress.cu
// and spmma.cu.
// 16-bit operands: 128 dense K per stage = 4 MMAs of K=32, metadata one TMEM column
// per MMA; FP8 operands: 256 dense K per stage = 4 MMAs of K=64, two columns per MMA.
// 8- and 4-bit integers run widened to bf16 on the 16-bit path, so they use its geometry.
// In both cases a stage of compressed A is 128 rows x 128 bytes, and the stage's
// metadata is one block [128 TMEM lanes][W words] (W = 4 for 16-bit, 8 for FP8): lane
// L's words for the stage's 4 MMAs in MMA order, which the GEMM's metadata writer warps
// store into the MMAs' TMEM slots.  The image is therefore the size of the canonical
// index (plus padding to whole tiles and stages).
constexpr int kBM = 128;
constexpr int kMmasPerStage = 4;
inline int stage_k(int t) { return is_f8(t) ? 256 : 128; }
inline int meta_lane_words(int t) { return is_f8(t) ? 8 : 4; }
inline int64_t meta_stage_bytes(int t) { return int64_t(kBM) * 4 * meta_lane_words(t); }
// The image covers whole 256-row tile pairs (the CTA-pair GEMM loads both halves).
inline int64_t meta_mtiles(int64_t M) { return 2 * ((M + 2 * kBM - 1) / (2 * kBM)); }

struct CompressArgs {
  const uint8_t* A; int64_t lda_bytes;
  const uint8_t* mask; int64_t ldm;
  uint8_t* values; int64_t ldv_bytes;
  uint32_t* index; int64_t ldi;
  int64_t M, K;
  int32_t* status;
  // fused compression + metadata image only: the image and its tiles / stages
  uint32_t* meta;
  int64_t mtiles, ksteps;
};

struct DecompressArgs {
  const uint8_t* values; int64_t ldv_bytes;
  const uint32_t* index; int64_t ldi;
  uint8_t* A; int64_t lda_bytes;
  int64_t M, K;
};

struct MetaArgs {
  const uint32_t* index; int64_t ldi;
  uint32_t* meta;
  int64_t M, K;       // dense sizes
  int64_t mtiles, ksteps;
};

cudaError_t launch_compress(const CompressArgs& a, int dtype, int mode, int num_sms, cudaStream_t s);
cudaError_t launch_compress_meta(const CompressArgs& a, int dtype, int mode, int num_sms,
                                 cudaStream_t s);
cudaError_t launch_decompress(const DecompressArgs& a, int dtype, int num_sms, cudaStream_t s);
cudaError_t launch_meta_prepare(const MetaArgs& a, int dtype, int num_sms, cudaStream_t s);
// rows x cols 8- or 4-bit integers (`bits`; pitch ld_src bytes) -> bfloat16 (pitch
// ld_dst elements)
cudaError_t launch_widen(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                         int64_t rows, int64_t cols, bool is_signed, int bits, int num_sms,
                         cudaStream_t s);

// Integer operands are widened to bf16 into a caller-provided workspace: A_c (M x K/2)
// then B (K x N, pitch rounded up to 8 elements).  Returns its size in bytes (0 for
// float operands).
int64_t int_ws_ldb(int64_t N);
size_t int_workspace_bytes(int64_t M, int64_t N, int64_t K);

// A strided batch of equal-shape problems: problem b's operands start at values +
// b * stride_values, meta + b * stride_meta (bytes), B + b * stride_b, C + b * stride_c,
// D + b * stride_d (elements of each operand's type).
struct BatchArgs {
  int64_t count;
  int64_t stride_values, stride_meta, stride_b, stride_c, stride_d;
};

// returns 0 on success, else an sp24_status value; batch == nullptr: one problem.
// index != nullptr (one problem only): the metadata comes from the canonical index
// (M x K/32 words, pitch ldi) and meta is not read.  diag_stall_ns != 0: the give-up
// self-test (the kernel's TMA producer issues no copies and every wait gives up after
// diag_stall_ns nanoseconds, setting the timeout bit of *status).
int launch_spmma(int ta, int tb, int tc, int td, int64_t M, int64_t N, int64_t K,
                 const void* values, int64_t ldv, const void* meta, const void* B, int64_t ldb,
                 const void* C, int64_t ldc, void* D, int64_t ldd, void* workspace,
                 int32_t* status, int num_sms, cudaStream_t s, const BatchArgs* batch = nullptr,
                 const uint32_t* index = nullptr, int64_t ldi = 0, uint64_t diag_stall_ns = 0);

// Up to kMaxGroupPerLaunch validated, non-empty float problems in one launch (the caller
// splits longer lists); returns 0 or an sp24_status value.
constexpr int kMaxGroupPerLaunch = 32;
int launch_spmma_grouped(int ta, int tb, int tc, int td, const sp24_mma_problem* problems,
                         int count, int32_t* status, int num_sms, cudaStream_t s);

// device properties of the current device, cached; returns false if not sm_103
bool current_device(int* num_sms);

}  // namespace sp24
