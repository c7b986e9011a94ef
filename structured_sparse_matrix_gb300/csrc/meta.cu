// meta.cu -- re-layout of the canonical sparsity index into the image from which the
// sparse GEMM fills, stage by stage, the metadata slots in tensor memory.
//
// Canonical index (as sp24_compress writes it): M x K/32 words, group g of row i in bits
// 4(g%8)..+3 of word g/8, nibble = p0 | p1 << 2.
//
// tcgen05.mma.sp reads the metadata of A from tensor memory (TMEM), one slot per MMA at
// a 16-column-aligned address.  In the GEMM four writer warps, one per quarter of the
// TMEM lanes, store each stage's words into the slots with tcgen05.st.  So the image
// holds, for every 128-row tile and every stage of the GEMM, one block
// [128 lanes][W words]: lane L's words for the stage's 4 MMAs, in MMA order (W = 4 for
// 16-bit types, W = 8 for FP8), read by the lane's thread with 16-byte loads.  It is a
// permutation of the canonical index plus padding: M x K / 8 bytes for whole tiles and
// stages.
//
// Word placement (measured on sm_103a with tcgen05.mma.sp, M = 128):
//   kind::f16 (16-bit types, 32 dense K per MMA, one word per lane): in each 16-row
//     band b, lane 16b+l holds the halves (h = l/8) of two rows' canonical words:
//       word = ((w[16b+l%8] >> 16h) & 0xffff) | ((w[16b+l%8+8] >> 16h) & 0xffff) << 16
//     so nibble q of lane 16b+l is group (q%4)+4h of row 16b+l%8+8(q/4).
//   kind::f8f6f4 (FP8 types, 64 dense K per MMA, two words per lane): lane = row, the
//     MMA's two words = the row's two canonical words of that K range, unchanged; the
//     lane's 8 words are thus the row's 8 canonical words of the stage in order.
//   8-bit and 4-bit integer types run widened to bf16 on kind::f16 and use its layout.
// The image covers M rounded up to a multiple of 256 and K to a multiple of the stage;
// rows beyond M and words beyond K/32 hold 0x44444444 (pattern {0,1} in every group).
// The matching values are zero, so they add nothing.
#include <cstdint>
#include <cuda_runtime.h>

#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {
namespace {

constexpr uint32_t kPadWord = 0x44444444u;

__device__ __forceinline__ uint32_t canon(const MetaArgs& a, int64_t row, int64_t w) {
  if (row >= a.M || w >= a.K / 32) return kPadWord;
  return a.index[row * a.ldi + w];
}

// Canonical words w0 .. w0+3 of one row: one 16-byte load when they are all inside the
// index and 16-byte aligned, else word by word with padding.
__device__ __forceinline__ uint4 canon4(const MetaArgs& a, int64_t row, int64_t w0) {
  const uint32_t* p = a.index + row * a.ldi + w0;
  if (row < a.M && w0 + 4 <= a.K / 32 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0)
    return __ldg(reinterpret_cast<const uint4*>(p));
  return make_uint4(canon(a, row, w0), canon(a, row, w0 + 1), canon(a, row, w0 + 2),
                    canon(a, row, w0 + 3));
}

// One thread per (tile, stage, lane): it reads the canonical words its lane needs and
// writes the lane's 16 (FP8: 32) bytes of the stage block, coalesced across a warp.
template <bool kEightBit>
__global__ void __launch_bounds__(256) meta_kernel(MetaArgs a) {
  griddep_launch_dependents();  // the GEMM after this pass may start its prologue
  const int64_t total = a.mtiles * a.ksteps * 128;
  for (int64_t o = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; o < total;
       o += int64_t(gridDim.x) * blockDim.x) {
    const int lane = int(o & 127);            // TMEM lane
    const int64_t blk = o >> 7;               // (mtile, kstep)
    const int64_t mt = blk / a.ksteps, ks = blk % a.ksteps;
    if constexpr (kEightBit) {
      const int64_t row = mt * 128 + lane;
      uint4* out = reinterpret_cast<uint4*>(a.meta) + (blk * 128 + lane) * 2;
      out[0] = canon4(a, row, ks * 8);
      out[1] = canon4(a, row, ks * 8 + 4);
    } else {
      const int band = lane >> 4, l = lane & 15;
      const int64_t rA = mt * 128 + band * 16 + (l & 7);
      const int h = l >> 3;
      const uint4 lo4 = canon4(a, rA, ks * 4), hi4 = canon4(a, rA + 8, ks * 4);
      const uint32_t lo[4] = {lo4.x, lo4.y, lo4.z, lo4.w}, hi[4] = {hi4.x, hi4.y, hi4.z, hi4.w};
      uint32_t w[kMmasPerStage];
#pragma unroll
      for (int j = 0; j < kMmasPerStage; ++j) {  // MMA j reads canonical word ks * 4 + j
        const uint32_t l16 = (lo[j] >> (16 * h)) & 0xFFFFu;
        const uint32_t h16 = (hi[j] >> (16 * h)) & 0xFFFFu;
        w[j] = l16 | (h16 << 16);
      }
      reinterpret_cast<uint4*>(a.meta)[blk * 128 + lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

}  // namespace

cudaError_t launch_meta_prepare(const MetaArgs& a, int dtype, int num_sms, cudaStream_t s) {
  const int64_t threads = a.mtiles * a.ksteps * 128;
  int64_t want = (threads + 255) / 256;
  int64_t cap = int64_t(num_sms) * 8;
  const int grid = int(want < cap ? (want > 0 ? want : 1) : cap);
  if (is_f8(dtype))
    meta_kernel<true><<<grid, 256, 0, s>>>(a);
  else
    meta_kernel<false><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sp24
