// api.cu -- the extern "C" entry points of libsp24 (declared in include/sp24.h):
// argument validation, device checks and stream-ordered launches.  No entry point
// allocates, frees or synchronises.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/sp24.h"
#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {

bool current_device(int* num_sms) {
  static std::mutex mu;
  static int cached_sms[64];
  static signed char cached_ok[64];  // 0 unknown, 1 sm_103, -1 other
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return false;
  }
  if (dev >= 64) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (cached_ok[dev] == 0) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    cached_ok[dev] = (major == 10 && minor == 3) ? 1 : -1;
    cached_sms[dev] = sms;
  }
  if (cached_ok[dev] != 1) return false;
  *num_sms = cached_sms[dev];
  return true;
}

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bounded-wait self-test: one thread waits on an mbarrier that nothing arrives at
__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  if (!mbar_wait(&bar, 0, &abort_flag, limit_ns)) atomicOr(status, kDevTimeout);
}

}  // namespace
}  // namespace sp24

using namespace sp24;

extern "C" {

int sp24_version(void) { return SP24_VERSION; }

const char* sp24_status_string(sp24_status s) {
  switch (s) {
    case SP24_OK: return "ok";
    case SP24_ERR_INVALID_ARG: return "invalid argument";
    case SP24_ERR_UNSUPPORTED: return "unsupported element-type combination";
    case SP24_ERR_ALIGN: return "pointer or row pitch not 16-byte aligned";
    case SP24_ERR_CUDA: return "CUDA error while enqueueing";
    case SP24_ERR_TIMEOUT: return "device wait timed out";
    case SP24_ERR_NOT_2_4: return "input is not 2:4 sparse";
    case SP24_ERR_NO_DEVICE: return "no sm_103 device is current";
    case SP24_ERR_SCRATCH_TOO_SMALL: return "problem needs more than the built-in scratch array";
    default: return "unknown status";
  }
}

sp24_status sp24_compress(sp24_dtype t, int64_t M, int64_t K, const void* A, int64_t lda,
                          const uint8_t* mask, int64_t ldm, sp24_mode mode, void* values,
                          int64_t ldv, uint32_t* index, int64_t ldi, int32_t* d_status,
                          void* stream) {
  if (!is_ab_type(t)) return SP24_ERR_UNSUPPORTED;
  if (mode < SP24_MODE_EXACT || mode > SP24_MODE_MAGNITUDE) return SP24_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return SP24_OK;
  if (!A || !values || !index || (mode == SP24_MODE_MASK && !mask)) return SP24_ERR_INVALID_ARG;
  if (lda < K || ldv < K / 2 || ldi < K / 32 || (mode == SP24_MODE_MASK && ldm < K))
    return SP24_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(values) || (reinterpret_cast<uintptr_t>(index) & 3u) ||
      !ld_ok16(t, lda) || !ld_ok16(t, ldv))
    return SP24_ERR_ALIGN;
  if (mode == SP24_MODE_MASK && (!aligned16(mask) || ldm % 16)) return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  CompressArgs a;
  a.A = static_cast<const uint8_t*>(A);
  a.lda_bytes = ld_bytes(t, lda);
  a.mask = mask;
  a.ldm = ldm;
  a.values = static_cast<uint8_t*>(values);
  a.ldv_bytes = ld_bytes(t, ldv);
  a.index = index;
  a.ldi = ldi;
  a.M = M;
  a.K = K;
  a.status = d_status;
  a.meta = nullptr;
  a.mtiles = a.ksteps = 0;
  if (launch_compress(a, t, mode, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SP24_ERR_CUDA;
  return SP24_OK;
}

sp24_status sp24_compress_meta(sp24_dtype t, int64_t M, int64_t K, const void* A, int64_t lda,
                               const uint8_t* mask, int64_t ldm, sp24_mode mode, void* values,
                               int64_t ldv, uint32_t* index, int64_t ldi, void* meta,
                               int32_t* d_status, void* stream) {
  if (!is_ab_type(t)) return SP24_ERR_UNSUPPORTED;
  if (mode < SP24_MODE_EXACT || mode > SP24_MODE_MAGNITUDE) return SP24_ERR_INVALID_ARG;
  if (M < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return SP24_OK;
  if (!A || !values || !meta || (mode == SP24_MODE_MASK && !mask)) return SP24_ERR_INVALID_ARG;
  if (lda < K || ldv < K / 2 || (index && ldi < K / 32) || (mode == SP24_MODE_MASK && ldm < K))
    return SP24_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(values) || !aligned16(meta) ||
      (reinterpret_cast<uintptr_t>(index) & 3u) || !ld_ok16(t, lda) || !ld_ok16(t, ldv))
    return SP24_ERR_ALIGN;
  if (mode == SP24_MODE_MASK && (!aligned16(mask) || ldm % 16)) return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  CompressArgs a;
  a.A = static_cast<const uint8_t*>(A);
  a.lda_bytes = ld_bytes(t, lda);
  a.mask = mask;
  a.ldm = ldm;
  a.values = static_cast<uint8_t*>(values);
  a.ldv_bytes = ld_bytes(t, ldv);
  a.index = index;
  a.ldi = ldi;
  a.M = M;
  a.K = K;
  a.status = d_status;
  a.meta = static_cast<uint32_t*>(meta);
  a.mtiles = meta_mtiles(M);
  a.ksteps = (K + stage_k(t) - 1) / stage_k(t);
  if (launch_compress_meta(a, t, mode, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SP24_ERR_CUDA;
  return SP24_OK;
}

sp24_status sp24_decompress(sp24_dtype t, int64_t M, int64_t K, const void* values,
                            int64_t ldv, const uint32_t* index, int64_t ldi, void* A,
                            int64_t lda, void* stream) {
  if (!is_ab_type(t)) return SP24_ERR_UNSUPPORTED;
  if (M < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return SP24_OK;
  if (!A || !values || !index) return SP24_ERR_INVALID_ARG;
  if (lda < K || ldv < K / 2 || ldi < K / 32) return SP24_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(values) || (reinterpret_cast<uintptr_t>(index) & 3u) ||
      !ld_ok16(t, lda) || !ld_ok16(t, ldv))
    return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  DecompressArgs a;
  a.values = static_cast<const uint8_t*>(values);
  a.ldv_bytes = ld_bytes(t, ldv);
  a.index = index;
  a.ldi = ldi;
  a.A = static_cast<uint8_t*>(A);
  a.lda_bytes = ld_bytes(t, lda);
  a.M = M;
  a.K = K;
  if (launch_decompress(a, t, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SP24_ERR_CUDA;
  return SP24_OK;
}

size_t sp24_meta_bytes(sp24_dtype t, int64_t M, int64_t K) {
  if (!is_ab_type(t) || M < 0 || K < 0 || (K % 32) != 0) return 0;
  const int64_t mtiles = meta_mtiles(M);
  const int64_t ksteps = (K + stage_k(t) - 1) / stage_k(t);
  return size_t(mtiles * ksteps * meta_stage_bytes(t));
}

sp24_status sp24_meta_prepare(sp24_dtype t, int64_t M, int64_t K, const uint32_t* index,
                              int64_t ldi, void* meta, void* stream) {
  if (!is_ab_type(t)) return SP24_ERR_UNSUPPORTED;
  if (M < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M == 0 || K == 0) return SP24_OK;
  if (!index || !meta || ldi < K / 32) return SP24_ERR_INVALID_ARG;
  if (!aligned16(meta) || (reinterpret_cast<uintptr_t>(index) & 3u)) return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  MetaArgs a;
  a.index = index;
  a.ldi = ldi;
  a.meta = static_cast<uint32_t*>(meta);
  a.M = M;
  a.K = K;
  a.mtiles = meta_mtiles(M);
  a.ksteps = (K + stage_k(t) - 1) / stage_k(t);
  if (launch_meta_prepare(a, t, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SP24_ERR_CUDA;
  return SP24_OK;
}

size_t sp24_mma_workspace_bytes(sp24_dtype ta, sp24_dtype tb, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  if ((is_i8(ta) && tb == SP24_S8) || (is_i4(ta) && is_i4(tb))) return int_workspace_bytes(M, N, K);
  return 0;
}

namespace {

// sp24_mma and sp24_mma_index: the product with the metadata from the image (meta) or
// from the canonical index (index != nullptr, pitch ldi words)
sp24_status mma_one(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td, int64_t M,
                    int64_t N, int64_t K, const void* values, int64_t ldv, const void* meta,
                    const uint32_t* index, int64_t ldi, const void* B, int64_t ldb,
                    const void* C, int64_t ldc, void* D, int64_t ldd, void* workspace,
                    size_t workspace_bytes, int32_t* d_status, void* stream) {
  const bool by_index = meta == nullptr;  // sp24_mma_index passes meta == nullptr
  const bool f16ish = (ta == SP24_F16 || ta == SP24_BF16);
  const bool f8 = is_f8(ta);
  const bool integer = is_int(ta);
  if (f16ish || f8) {
    // 16-bit: A and B of one type; FP8: any mix of E4M3 and E5M2 (kind::f8f6f4 takes
    // separate A and B type fields).  C and D: f32, bf16 or f16 each.
    if (f16ish ? tb != ta : !is_f8(tb)) return SP24_ERR_UNSUPPORTED;
    if (C != nullptr && !is_float_acc(tc)) return SP24_ERR_UNSUPPORTED;
    if (!is_float_acc(td)) return SP24_ERR_UNSUPPORTED;
  } else if (integer) {
    // 8-bit: B signed (u8 x u8 products could leave an f32 chunk sum inexact); 4-bit: any
    // mix of signed and unsigned
    if (is_i8(ta) ? tb != SP24_S8 : !is_i4(tb)) return SP24_ERR_UNSUPPORTED;
    if (C != nullptr && tc != SP24_S32) return SP24_ERR_UNSUPPORTED;
    if (td != SP24_S32) return SP24_ERR_UNSUPPORTED;
  } else {
    return SP24_ERR_UNSUPPORTED;
  }
  if (M < 0 || N < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return SP24_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SP24_OK;
  if (!D || (K > 0 && (!values || !B || (by_index ? !index : !meta))))
    return SP24_ERR_INVALID_ARG;
  if (ldd < N || (C && ldc < N) || (K > 0 && (ldv < K / 2 || ldb < N))) return SP24_ERR_INVALID_ARG;
  if (by_index && K > 0 && ldi < K / 32) return SP24_ERR_INVALID_ARG;
  if (integer && K > 0 && (!workspace || workspace_bytes < int_workspace_bytes(M, N, K)))
    return SP24_ERR_INVALID_ARG;
  const int dsz = dtype_bytes(td);
  if (!aligned16(D) || (ldd * dsz) % 16) return SP24_ERR_ALIGN;
  if (C && (!aligned16(C) || (ldc * dtype_bytes(tc)) % 16)) return SP24_ERR_ALIGN;
  if (K > 0 && (!aligned16(values) || !aligned16(B) || !ld_ok16(ta, ldv) || !ld_ok16(tb, ldb)))
    return SP24_ERR_ALIGN;
  if (K > 0 && (by_index ? (reinterpret_cast<uintptr_t>(index) & 3u) != 0 : !aligned16(meta)))
    return SP24_ERR_ALIGN;
  if (integer && K > 0 && !aligned16(workspace)) return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  const int rc = launch_spmma(ta, tb, tc, td, M, N, K, values, ldv, by_index ? nullptr : meta, B,
                              ldb, C, ldc, D, ldd, workspace, d_status, sms,
                              static_cast<cudaStream_t>(stream), nullptr,
                              (by_index && K > 0) ? index : nullptr, ldi);
  return static_cast<sp24_status>(rc);
}

}  // namespace

sp24_status sp24_mma(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td, int64_t M,
                     int64_t N, int64_t K, const void* values, int64_t ldv, const void* meta,
                     const void* B, int64_t ldb, const void* C, int64_t ldc, void* D,
                     int64_t ldd, void* workspace, size_t workspace_bytes, int32_t* d_status,
                     void* stream) {
  return mma_one(ta, tb, tc, td, M, N, K, values, ldv, meta, nullptr, 0, B, ldb, C, ldc, D, ldd,
                 workspace, workspace_bytes, d_status, stream);
}

sp24_status sp24_mma_index(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td,
                           int64_t M, int64_t N, int64_t K, const void* values, int64_t ldv,
                           const uint32_t* index, int64_t ldi, const void* B, int64_t ldb,
                           const void* C, int64_t ldc, void* D, int64_t ldd, void* workspace,
                           size_t workspace_bytes, int32_t* d_status, void* stream) {
  return mma_one(ta, tb, tc, td, M, N, K, values, ldv, nullptr, index, ldi, B, ldb, C, ldc, D,
                 ldd, workspace, workspace_bytes, d_status, stream);
}

sp24_status sp24_mma_strided_batched(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc,
                                     sp24_dtype td, int64_t batch, int64_t M, int64_t N,
                                     int64_t K, const void* values, int64_t ldv,
                                     int64_t stride_values, const void* meta,
                                     int64_t stride_meta, const void* B, int64_t ldb,
                                     int64_t stride_b, const void* C, int64_t ldc,
                                     int64_t stride_c, void* D, int64_t ldd, int64_t stride_d,
                                     int32_t* d_status, void* stream) {
  const bool f16ish = (ta == SP24_F16 || ta == SP24_BF16);
  if (!(f16ish || is_f8(ta))) return SP24_ERR_UNSUPPORTED;  // float operands only
  if (f16ish ? tb != ta : !is_f8(tb)) return SP24_ERR_UNSUPPORTED;
  if (C != nullptr && !is_float_acc(tc)) return SP24_ERR_UNSUPPORTED;
  if (!is_float_acc(td)) return SP24_ERR_UNSUPPORTED;
  if (batch < 0 || M < 0 || N < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return SP24_ERR_INVALID_ARG;
  if (batch == 0 || M == 0 || N == 0) return SP24_OK;
  // every tile of the launch is numbered with an int
  if ((M + 127) / 128 * ((N + 31) / 32) * batch > INT32_MAX / 2) return SP24_ERR_INVALID_ARG;
  if (!D || (K > 0 && (!values || !meta || !B))) return SP24_ERR_INVALID_ARG;
  if (ldd < N || (C && ldc < N) || (K > 0 && (ldv < K / 2 || ldb < N))) return SP24_ERR_INVALID_ARG;
  const int esz = dtype_bytes(ta);
  const int dsz = dtype_bytes(td);
  if (batch > 1) {
    // D of different problems must not overlap; the operands are only read
    if (stride_d < M * ldd) return SP24_ERR_INVALID_ARG;
    if (C && stride_c < 0) return SP24_ERR_INVALID_ARG;
    if (K > 0 && (stride_values < 0 || stride_b < 0 ||
                  size_t(stride_meta) < sp24_meta_bytes(ta, M, K)))
      return SP24_ERR_INVALID_ARG;
    if ((stride_d * dsz) % 16 || (C && (stride_c * dtype_bytes(tc)) % 16)) return SP24_ERR_ALIGN;
    if (K > 0 && ((stride_values * esz) % 16 || (stride_b * esz) % 16 || stride_meta % 16))
      return SP24_ERR_ALIGN;
  }
  if (!aligned16(D) || (ldd * dsz) % 16) return SP24_ERR_ALIGN;
  if (C && (!aligned16(C) || (ldc * dtype_bytes(tc)) % 16)) return SP24_ERR_ALIGN;
  if (K > 0 && (!aligned16(values) || !aligned16(meta) || !aligned16(B) || (ldv * esz) % 16 ||
                (ldb * esz) % 16))
    return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  BatchArgs ba;
  ba.count = batch;
  ba.stride_values = stride_values;
  ba.stride_meta = stride_meta;
  ba.stride_b = stride_b;
  ba.stride_c = stride_c;
  ba.stride_d = stride_d;
  const int rc = launch_spmma(ta, tb, tc, td, M, N, K, values, ldv, meta, B, ldb, C, ldc, D, ldd,
                              nullptr, d_status, sms, static_cast<cudaStream_t>(stream), &ba);
  return static_cast<sp24_status>(rc);
}

sp24_status sp24_mma_grouped(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc, sp24_dtype td,
                             const sp24_mma_problem* problems, int64_t count, int32_t* d_status,
                             void* stream) {
  const bool f16ish = (ta == SP24_F16 || ta == SP24_BF16);
  if (!(f16ish || is_f8(ta))) return SP24_ERR_UNSUPPORTED;  // float operands only
  if (f16ish ? tb != ta : !is_f8(tb)) return SP24_ERR_UNSUPPORTED;
  if (!is_float_acc(tc) || !is_float_acc(td)) return SP24_ERR_UNSUPPORTED;
  if (count < 0 || (count > 0 && !problems)) return SP24_ERR_INVALID_ARG;
  const int esz = dtype_bytes(ta);
  const int dsz = dtype_bytes(td);
  const int csz = dtype_bytes(tc);
  int64_t live = 0;
  for (int64_t g = 0; g < count; ++g) {
    const sp24_mma_problem& q = problems[g];
    if (q.M < 0 || q.N < 0 || q.K < 0 || (q.K % 32) != 0) return SP24_ERR_INVALID_ARG;
    if (q.M > INT32_MAX / 2 || q.N > INT32_MAX / 2 || q.K > INT32_MAX / 2)
      return SP24_ERR_INVALID_ARG;
    if (q.M == 0 || q.N == 0) continue;
    if (!q.D || (q.K > 0 && (!q.values || !q.meta || !q.B))) return SP24_ERR_INVALID_ARG;
    if (q.ldd < q.N || (q.C && q.ldc < q.N) || (q.K > 0 && (q.ldv < q.K / 2 || q.ldb < q.N)))
      return SP24_ERR_INVALID_ARG;
    if ((q.M + 255) / 256 * ((q.N + 31) / 32) > INT32_MAX / 64) return SP24_ERR_INVALID_ARG;
    if (!aligned16(q.D) || (q.ldd * dsz) % 16) return SP24_ERR_ALIGN;
    if (q.C && (!aligned16(q.C) || (q.ldc * csz) % 16)) return SP24_ERR_ALIGN;
    if (q.K > 0 && (!aligned16(q.values) || !aligned16(q.meta) || !aligned16(q.B) ||
                    (q.ldv * esz) % 16 || (q.ldb * esz) % 16))
      return SP24_ERR_ALIGN;
    ++live;
  }
  if (live == 0) return SP24_OK;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  // launches of up to kMaxGroupPerLaunch non-empty problems, in order
  sp24_mma_problem batch[kMaxGroupPerLaunch];
  int n = 0;
  for (int64_t g = 0; g <= count; ++g) {
    if (g < count && problems[g].M > 0 && problems[g].N > 0) batch[n++] = problems[g];
    if (n == kMaxGroupPerLaunch || (g == count && n > 0)) {
      const int rc = launch_spmma_grouped(ta, tb, tc, td, batch, n, d_status, sms,
                                          static_cast<cudaStream_t>(stream));
      if (rc != 0) return static_cast<sp24_status>(rc);
      n = 0;
    }
  }
  return SP24_OK;
}

sp24_status sp24_diag_mma_stall(sp24_dtype ta, int64_t M, int64_t N, int64_t K,
                                const void* values, int64_t ldv, const void* meta, const void* B,
                                int64_t ldb, void* D, int64_t ldd, uint64_t limit_ns,
                                int32_t* d_status, void* stream) {
  if (!(ta == SP24_F16 || ta == SP24_BF16 || is_f8(ta))) return SP24_ERR_UNSUPPORTED;
  if (!d_status || limit_ns == 0 || limit_ns > 1000000000ull) return SP24_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return SP24_ERR_INVALID_ARG;
  if (!values || !meta || !B || !D) return SP24_ERR_INVALID_ARG;
  if (ldd < N || ldv < K / 2 || ldb < N) return SP24_ERR_INVALID_ARG;
  if (!aligned16(D) || (ldd * 4) % 16 || !aligned16(values) || !aligned16(B) ||
      !aligned16(meta) || !ld_ok16(ta, ldv) || !ld_ok16(ta, ldb))
    return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  const int rc = launch_spmma(ta, ta, SP24_F32, SP24_F32, M, N, K, values, ldv, meta, B, ldb,
                              nullptr, N, D, ldd, nullptr, d_status, sms,
                              static_cast<cudaStream_t>(stream), nullptr, nullptr, 0, limit_ns);
  return static_cast<sp24_status>(rc);
}

sp24_status sp24_diag_wait_timeout(int32_t* d_status, uint64_t limit_ns, void* stream) {
  if (!d_status) return SP24_ERR_INVALID_ARG;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  wait_timeout_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(d_status, limit_ns);
  return cudaGetLastError() == cudaSuccess ? SP24_OK : SP24_ERR_CUDA;
}

}  // extern "C"
