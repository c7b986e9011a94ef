// compress.cu -- 2:4 compression (exact / mask / magnitude) and decompression kernels.
//
// What is computed ("RDNA4 sparse WMMA builtins", "Structured sparsity (2:4 pattern)":
// walk K in groups of four, keep the two non-zero positions, pack them consecutively;
// "CDNA and CDNA2 sparse MFMA builtins": index literal 0x88 for positions {0, 2}):
//   values[i][2g], values[i][2g+1] = A[i][4g+p0], A[i][4g+p1]   (p0 < p1, bit copies)
//   index[i][g/8] bits 4(g%8)..+3  = p0 | p1 << 2
//
// Layout of the work: one thread owns one 16-byte chunk of a row of A (8 elements of a
// 16-bit type = 2 groups, or 16 elements of an 8-bit type = 4 groups).  A warp owns 32
// consecutive chunks, so every load of A and every store of values is a fully
// coalesced 16- / 8-byte vector access; the 4 (16-bit) or 2 (8-bit) lanes that share
// one 32-element index word merge their nibbles with two / one xor-shuffles.  The
// kernel is HBM-bound: it streams A (+ mask) once and writes values + index once.
#include <cstdint>
#include <cuda_runtime.h>

#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {
namespace {

// element classes: how "zero" and "|x|" are read from the stored bits
enum ElemClass { kFloat16 = 0, kFloat8 = 1, kSigned8 = 2, kUnsigned8 = 3 };

template <int CLS>
__device__ __forceinline__ uint32_t magnitude_key(uint32_t b) {
  if constexpr (CLS == kFloat16) return b & 0x7FFFu;  // sign cleared: orders |x|
  if constexpr (CLS == kFloat8) return b & 0x7Fu;
  if constexpr (CLS == kSigned8) {
    int v = static_cast<int8_t>(static_cast<uint8_t>(b));
    return static_cast<uint32_t>(v < 0 ? -v : v);
  }
  return b & 0xFFu;
}

template <int CLS>
__device__ __forceinline__ bool is_nonzero(uint32_t b) {
  if constexpr (CLS == kFloat16) return (b & 0x7FFFu) != 0u;  // +0 and -0 are zero
  if constexpr (CLS == kFloat8) return (b & 0x7Fu) != 0u;
  return (b & 0xFFu) != 0u;
}

// Choose (p0, p1) for one group.  keep: 4-bit set of candidate positions (exact / mask
// modes).  Returns the nibble and sets *flag when the group breaks the 2:4 rule.
__device__ __forceinline__ uint32_t pick_from_set(uint32_t keep, bool mask_mode, bool* flag) {
  const int n = __popc(keep);
  *flag = mask_mode ? (n != 2) : (n > 2);
  uint32_t s = keep;
  if (n > 2) {  // keep the two lowest
    uint32_t lo = s & (0u - s);
    uint32_t rest = s ^ lo;
    s = lo | (rest & (0u - rest));
  }
  while (__popc(s) < 2) s |= (~s) & (s + 1u);  // add the lowest free position
  const uint32_t p0 = __ffs(s) - 1;
  const uint32_t p1 = 31 - __clz(s);
  return p0 | (p1 << 2);
}

// x[i] for a run-time i in 0..3 without indexing memory (keeps x in registers)
__device__ __forceinline__ uint32_t sel4(const uint32_t (&x)[4], uint32_t i) {
  const uint32_t lo = (i & 1u) ? x[1] : x[0];
  const uint32_t hi = (i & 1u) ? x[3] : x[2];
  return (i & 2u) ? hi : lo;
}

template <int CLS>
__device__ __forceinline__ uint32_t pick_magnitude(const uint32_t (&x)[4]) {
  uint32_t k[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) k[p] = magnitude_key<CLS>(x[p]);
  int best = 0;
#pragma unroll
  for (int p = 1; p < 4; ++p)
    if (k[p] > k[best]) best = p;  // strict: equal keys keep the lower position
  int second = best == 0 ? 1 : 0;
#pragma unroll
  for (int p = 0; p < 4; ++p)
    if (p != best && k[p] > k[second]) second = p;
  const uint32_t p0 = best < second ? best : second;
  const uint32_t p1 = best < second ? second : best;
  return p0 | (p1 << 2);
}

// ESZ = element bytes (2 or 1); MODE = SP24_MODE_* value.  Each warp step covers kUnroll
// groups of 32 consecutive chunks; all their loads are issued before any is used, so a
// thread keeps kUnroll 16-byte loads (plus mask loads) in flight.
template <int ESZ, int CLS, int MODE>
__global__ void __launch_bounds__(256) compress_kernel(CompressArgs a) {
  constexpr int kElems = 16 / ESZ;   // elements per 16-byte chunk
  constexpr int kGroups = kElems / 4;  // groups per chunk
  constexpr int kLanesPerWord = 32 / kElems;
  constexpr int kUnroll = 4;
  const int lane = threadIdx.x & 31;
  const int64_t cpr = a.K / kElems;  // chunks per row
  const int64_t total = a.M * cpr;
  const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t warp_stride = (int64_t(gridDim.x) * blockDim.x) >> 5;
  bool any_flag = false;

  for (int64_t base = warp_global * 32 * kUnroll; base < total;
       base += warp_stride * 32 * kUnroll) {
    uint4 v[kUnroll];
    uint32_t mbits[kUnroll][4];
    int64_t row[kUnroll], cc[kUnroll];
    bool active[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * 32 + lane;
      active[u] = c < total;
      row[u] = active[u] ? c / cpr : 0;
      cc[u] = active[u] ? c - row[u] * cpr : 0;
      v[u] = make_uint4(0, 0, 0, 0);
      mbits[u][0] = mbits[u][1] = mbits[u][2] = mbits[u][3] = 0;
      if (active[u]) {
        v[u] = __ldcs(reinterpret_cast<const uint4*>(a.A + row[u] * a.lda_bytes + cc[u] * 16));
        if constexpr (MODE == 1) {
          if constexpr (kElems == 8) {
            const uint2 m =
                __ldcs(reinterpret_cast<const uint2*>(a.mask + row[u] * a.ldm + cc[u] * 8));
            mbits[u][0] = m.x;
            mbits[u][1] = m.y;
          } else {
            const uint4 m =
                __ldcs(reinterpret_cast<const uint4*>(a.mask + row[u] * a.ldm + cc[u] * 16));
            mbits[u][0] = m.x;
            mbits[u][1] = m.y;
            mbits[u][2] = m.z;
            mbits[u][3] = m.w;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t out[2] = {0, 0};  // kept elements, packed
      uint32_t nibs = 0;
#pragma unroll
      for (int g = 0; g < kGroups; ++g) {
        uint32_t x[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int e = 4 * g + p;  // element index within the chunk
          if constexpr (ESZ == 2)
            x[p] = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
          else
            x[p] = (w[e >> 2] >> (8 * (e & 3))) & 0xFFu;
        }
        uint32_t nib;
        bool flag = false;
        if constexpr (MODE == 2) {
          nib = pick_magnitude<CLS>(x);
        } else {
          uint32_t keep = 0;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            bool k;
            if constexpr (MODE == 1) {
              const int e = 4 * g + p;
              k = ((mbits[u][e >> 2] >> (8 * (e & 3))) & 0xFFu) != 0u;
            } else {
              k = is_nonzero<CLS>(x[p]);
            }
            keep |= uint32_t(k) << p;
          }
          nib = pick_from_set(keep, MODE == 1, &flag);
        }
        any_flag |= (flag && active[u]);
        const uint32_t k0 = sel4(x, nib & 3u), k1 = sel4(x, nib >> 2);
        if constexpr (ESZ == 2) {
          out[g] = k0 | (k1 << 16);
        } else {
          out[g >> 1] |= (k0 | (k1 << 8)) << (16 * (g & 1));
        }
        nibs |= nib << (4 * g);
      }
      if (active[u]) {
        __stcs(reinterpret_cast<uint2*>(a.values + row[u] * a.ldv_bytes + cc[u] * 8),
               make_uint2(out[0], out[1]));
      }
      // merge the nibbles of the lanes that share one index word
      uint32_t word = nibs << ((4 * kGroups) * (lane % kLanesPerWord));
#pragma unroll
      for (int o = 1; o < kLanesPerWord; o <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, o);
      if (active[u] && (lane % kLanesPerWord) == 0) {
        a.index[row[u] * a.ldi + (cc[u] * kElems) / 32] = word;
      }
    }
  }
  if (a.status != nullptr && __any_sync(0xFFFFFFFFu, any_flag) && lane == 0)
    atomicOr(a.status, kDevNot24);
}

// expand(values, index): one thread writes one 16-byte chunk of dense A.
template <int ESZ>
__global__ void __launch_bounds__(256) decompress_kernel(DecompressArgs a) {
  constexpr int kElems = 16 / ESZ;
  constexpr int kGroups = kElems / 4;
  const int64_t cpr = a.K / kElems;
  const int64_t total = a.M * cpr;
  for (int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; c < total;
       c += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = c / cpr, cc = c - row * cpr;
    const uint2 vv = *reinterpret_cast<const uint2*>(a.values + row * a.ldv_bytes + cc * 8);
    const uint32_t word = a.index[row * a.ldi + (cc * kElems) / 32];
    const uint32_t nibs = word >> ((cc * kElems) % 32) / 4 * 4;
    uint32_t o[4] = {0, 0, 0, 0};
    const uint32_t kv[2] = {vv.x, vv.y};
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const uint32_t nib = (nibs >> (4 * g)) & 0xFu;
      const uint32_t p0 = nib & 3u, p1 = nib >> 2;
      uint32_t k0, k1;
      if constexpr (ESZ == 2) {
        k0 = kv[g] & 0xFFFFu;
        k1 = kv[g] >> 16;
      } else {
        const uint32_t h = (kv[g >> 1] >> (16 * (g & 1))) & 0xFFFFu;
        k0 = h & 0xFFu;
        k1 = h >> 8;
      }
      const int e0 = 4 * g + p0, e1 = 4 * g + p1;
      if constexpr (ESZ == 2) {
        o[e0 >> 1] |= k0 << (16 * (e0 & 1));
        o[e1 >> 1] |= k1 << (16 * (e1 & 1));
      } else {
        o[e0 >> 2] |= k0 << (8 * (e0 & 3));
        o[e1 >> 2] |= k1 << (8 * (e1 & 3));
      }
    }
    *reinterpret_cast<uint4*>(a.A + row * a.lda_bytes + cc * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int ESZ, int CLS>
cudaError_t launch_compress_cls(const CompressArgs& a, int mode, int grid, cudaStream_t s) {
  switch (mode) {
    case 0: compress_kernel<ESZ, CLS, 0><<<grid, 256, 0, s>>>(a); break;
    case 1: compress_kernel<ESZ, CLS, 1><<<grid, 256, 0, s>>>(a); break;
    default: compress_kernel<ESZ, CLS, 2><<<grid, 256, 0, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, int dtype, int mode, int num_sms,
                            cudaStream_t s) {
  const int esz = dtype_bytes(dtype);
  const int64_t chunks = a.M * (a.K / (16 / esz));
  // each thread covers 4 chunks per step; 8 resident blocks of 256 threads per SM
  int64_t want = (chunks + 1023) / 1024;
  int64_t cap = int64_t(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
  switch (dtype) {
    case kF16:
    case kBF16: return launch_compress_cls<2, kFloat16>(a, mode, grid, s);
    case kE4M3:
    case kE5M2: return launch_compress_cls<1, kFloat8>(a, mode, grid, s);
    case kS8: return launch_compress_cls<1, kSigned8>(a, mode, grid, s);
    default: return launch_compress_cls<1, kUnsigned8>(a, mode, grid, s);
  }
}

cudaError_t launch_decompress(const DecompressArgs& a, int dtype, int num_sms, cudaStream_t s) {
  const int esz = dtype_bytes(dtype);
  const int64_t chunks = a.M * (a.K / (16 / esz));
  int64_t want = (chunks + 255) / 256;
  int64_t cap = int64_t(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
  if (esz == 2)
    decompress_kernel<2><<<grid, 256, 0, s>>>(a);
  else
    decompress_kernel<1><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sp24
