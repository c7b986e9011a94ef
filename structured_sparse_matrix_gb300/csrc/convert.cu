// convert.cu -- exact widening of 8-bit integer operands to bfloat16 for the integer path
// of the sparse GEMM.
//
// Every signed (-128..127) and unsigned (0..255) 8-bit integer is exactly representable in
// bfloat16 (8 significant bits), so the integer product can run on the bf16 sparse tensor
// cores without rounding ("RDNA4 dense WMMA builtins", "Common parameters": a_neg / b_neg
// choose signed or unsigned operands).  One thread widens 16 bytes (one vector load) into
// 32 bytes (two vector stores); rows keep their own pitch on each side.  HBM-bound.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "sp24_internal.h"

namespace sp24 {
namespace {

template <bool kSigned>
__global__ void __launch_bounds__(256) widen_kernel(const uint8_t* src, int64_t ld_src,
                                                    __nv_bfloat16* dst, int64_t ld_dst,
                                                    int64_t rows, int64_t cols) {
  const int64_t cpr = (cols + 15) / 16;  // 16-byte chunks per row (last one may be partial)
  const int64_t total = rows * cpr;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = c / cpr, k = (c - r * cpr) * 16;
    if (k + 16 > cols) {  // ragged tail: element by element, never past `cols`
      for (int64_t j = k; j < cols; ++j) {
        const uint32_t b = src[r * ld_src + j];
        dst[r * ld_dst + j] = __float2bfloat16_rn(kSigned ? float(int8_t(uint8_t(b))) : float(b));
      }
      continue;
    }
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src + r * ld_src + k));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t b0 = (w[i >> 1] >> (16 * (i & 1))) & 0xFFu;
      const uint32_t b1 = (w[i >> 1] >> (16 * (i & 1) + 8)) & 0xFFu;
      const float f0 = kSigned ? float(int8_t(uint8_t(b0))) : float(b0);
      const float f1 = kSigned ? float(int8_t(uint8_t(b1))) : float(b1);
      __nv_bfloat162 h = __floats2bfloat162_rn(f0, f1);  // exact: |x| <= 255
      memcpy(&o[i], &h, 4);
    }
    uint4* d = reinterpret_cast<uint4*>(dst + r * ld_dst + k);
    __stcs(d, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(d + 1, make_uint4(o[4], o[5], o[6], o[7]));
  }
}

}  // namespace

cudaError_t launch_widen(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                         int64_t rows, int64_t cols, bool is_signed, int num_sms,
                         cudaStream_t s) {
  const int64_t chunks = rows * ((cols + 15) / 16);
  int64_t want = (chunks + 255) / 256;
  const int64_t cap = int64_t(num_sms) * 8;
  const int grid = int(want < cap ? (want > 0 ? want : 1) : cap);
  auto d = static_cast<__nv_bfloat16*>(dst);
  auto sp = static_cast<const uint8_t*>(src);
  if (is_signed)
    widen_kernel<true><<<grid, 256, 0, s>>>(sp, ld_src, d, ld_dst, rows, cols);
  else
    widen_kernel<false><<<grid, 256, 0, s>>>(sp, ld_src, d, ld_dst, rows, cols);
  return cudaGetLastError();
}

}  // namespace sp24
