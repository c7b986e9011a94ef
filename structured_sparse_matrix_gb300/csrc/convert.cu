// convert.cu -- exact widening of 8- and 4-bit integer operands to bfloat16 for the
// integer path of the sparse GEMM.
//
// Every signed (-128..127) and unsigned (0..255) 8-bit integer, and so every 4-bit one
// (-8..7, 0..15), is exactly representable in bfloat16 (8 significant bits), so the
// integer product can run on the bf16 sparse tensor cores without rounding ("RDNA4 dense
// WMMA builtins", "Common parameters": a_neg / b_neg choose signed or unsigned operands;
// "RDNA4 sparse WMMA builtins", "INT4 and UINT4 inputs": two 4-bit elements per byte).
// One thread widens 16 elements (one 16- or 8-byte vector load) into 32 bytes (two
// vector stores); rows keep their own pitch on each side.  HBM-bound.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {
namespace {

// the integer value of a kBits-wide field x (two's complement if kSigned)
template <bool kSigned, int kBits>
__device__ __forceinline__ float int_value(uint32_t x) {
  if constexpr (kSigned) return float(int(x) - int((x & (1u << (kBits - 1))) << 1));
  return float(x);
}

// element j of a row: 8-bit -> byte j; 4-bit -> byte j/2, low nibble for even j
template <int kBits>
__device__ __forceinline__ uint32_t field(const uint8_t* row, int64_t j) {
  if constexpr (kBits == 8) return row[j];
  return (row[j >> 1] >> (4 * (j & 1))) & 0xFu;
}

template <bool kSigned, int kBits>
__global__ void __launch_bounds__(256) widen_kernel(const uint8_t* src, int64_t ld_src,
                                                    __nv_bfloat16* dst, int64_t ld_dst,
                                                    int64_t rows, int64_t cols) {
  griddep_launch_dependents();  // the GEMM after this pass may start its prologue
  constexpr uint32_t kMask = (1u << kBits) - 1;
  const int64_t cpr = (cols + 15) / 16;  // 16-element chunks per row (last may be partial)
  const int64_t total = rows * cpr;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += int64_t(gridDim.x) * blockDim.x) {
    const int64_t r = c / cpr, k = (c - r * cpr) * 16;
    if (k + 16 > cols) {  // ragged tail: element by element, never past `cols`
      for (int64_t j = k; j < cols; ++j)
        dst[r * ld_dst + j] =
            __float2bfloat16_rn(int_value<kSigned, kBits>(field<kBits>(src + r * ld_src, j)));
      continue;
    }
    uint32_t w[4];
    if constexpr (kBits == 8) {
      const uint4 v = __ldcs(reinterpret_cast<const uint4*>(src + r * ld_src + k));
      w[0] = v.x, w[1] = v.y, w[2] = v.z, w[3] = v.w;
    } else {
      const uint2 v = __ldcs(reinterpret_cast<const uint2*>(src + r * ld_src + k / 2));
      w[0] = v.x, w[1] = v.y, w[2] = w[3] = 0;
    }
    uint32_t o[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {  // elements 2i, 2i+1
      const int b = 2 * i * kBits;  // bit offset of element 2i in w
      const uint32_t x0 = (w[b >> 5] >> (b & 31)) & kMask;
      const uint32_t x1 = (w[b >> 5] >> ((b & 31) + kBits)) & kMask;
      __nv_bfloat162 h = __floats2bfloat162_rn(int_value<kSigned, kBits>(x0),
                                               int_value<kSigned, kBits>(x1));  // exact
      memcpy(&o[i], &h, 4);
    }
    uint4* d = reinterpret_cast<uint4*>(dst + r * ld_dst + k);
    __stcs(d, make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(d + 1, make_uint4(o[4], o[5], o[6], o[7]));
  }
}

}  // namespace

cudaError_t launch_widen(const void* src, int64_t ld_src, void* dst, int64_t ld_dst,
                         int64_t rows, int64_t cols, bool is_signed, int bits, int num_sms,
                         cudaStream_t s) {
  const int64_t chunks = rows * ((cols + 15) / 16);
  int64_t want = (chunks + 255) / 256;
  const int64_t cap = int64_t(num_sms) * 8;
  const int grid = int(want < cap ? (want > 0 ? want : 1) : cap);
  auto d = static_cast<__nv_bfloat16*>(dst);
  auto sp = static_cast<const uint8_t*>(src);
  if (bits == 8) {
    if (is_signed)
      widen_kernel<true, 8><<<grid, 256, 0, s>>>(sp, ld_src, d, ld_dst, rows, cols);
    else
      widen_kernel<false, 8><<<grid, 256, 0, s>>>(sp, ld_src, d, ld_dst, rows, cols);
  } else {
    if (is_signed)
      widen_kernel<true, 4><<<grid, 256, 0, s>>>(sp, ld_src, d, ld_dst, rows, cols);
    else
      widen_kernel<false, 4><<<grid, 256, 0, s>>>(sp, ld_src, d, ld_dst, rows, cols);
  }
  return cudaGetLastError();
}

}  // namespace sp24
