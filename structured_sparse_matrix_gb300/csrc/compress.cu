// compress.cu -- 2:4 compression (exact / mask / magnitude) and decompression kernels.
//
// What is computed ("RDNA4 sparse WMMA builtins", "Structured sparsity (2:4 pattern)":
// walk K in groups of four, keep the two non-zero positions, pack them consecutively;
// "CDNA and CDNA2 sparse MFMA builtins": index literal 0x88 for positions {0, 2}):
//   values[i][2g], values[i][2g+1] = A[i][4g+p0], A[i][4g+p1]   (p0 < p1, bit copies)
//   index[i][g/8] bits 4(g%8)..+3  = p0 | p1 << 2
//
// Layout of the work: one thread owns one 16-byte chunk of a row of A (8 elements of a
// 16-bit type = 2 groups, 16 elements of an 8-bit type = 4 groups, or 32 elements of a
// 4-bit type = 8 groups, two per byte with element 2i in the low nibble as in "INT4 and
// UINT4 inputs").  A warp owns 32 consecutive chunks, so every load of A and every store
// of values is a fully coalesced 16- / 8-byte vector access; the 4 (16-bit) or 2 (8-bit)
// lanes that share one 32-element index word merge their nibbles with two / one
// xor-shuffles (a 4-bit chunk fills a word alone).  The kernel is HBM-bound: it streams
// A (+ mask) once and writes values + index once.
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>

#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {
namespace {

// element classes: how "zero" and "|x|" are read from the stored bits
enum ElemClass { kFloat16 = 0, kFloat8 = 1, kSigned8 = 2, kUnsigned8 = 3, kSigned4 = 4,
                 kUnsigned4 = 5 };

// Selection rule of the exact and mask modes as a function of the 4-bit set of candidate
// positions: more than two -> the two lowest; fewer than two -> add the lowest free
// positions until there are two.  kPickLut holds the resulting nibble p0 | p1 << 2 for
// every set (4 bits each); kFlagMask / kFlagExact have bit `set` on when the group
// breaks the rule of that mode (mask: not exactly two; exact: more than two).
constexpr uint32_t pick_rule(uint32_t keep) {
  uint32_t s = keep;
  int n = 0;
  for (int p = 0; p < 4; ++p) n += (s >> p) & 1u;
  if (n > 2) {
    const uint32_t lo = s & (0u - s);
    const uint32_t rest = s ^ lo;
    s = lo | (rest & (0u - rest));
  }
  for (int p = 0; p < 4 && n < 2; ++p)
    if (!((s >> p) & 1u)) {
      s |= 1u << p;
      ++n;
    }
  uint32_t p0 = 0, p1 = 0;
  for (int p = 3; p >= 0; --p)
    if ((s >> p) & 1u) p0 = uint32_t(p);
  for (int p = 0; p < 4; ++p)
    if ((s >> p) & 1u) p1 = uint32_t(p);
  return p0 | (p1 << 2);
}
constexpr uint64_t make_pick_lut() {
  uint64_t r = 0;
  for (uint32_t k = 0; k < 16; ++k) r |= uint64_t(pick_rule(k)) << (4 * k);
  return r;
}
constexpr uint32_t make_flag_lut(bool mask_mode) {
  uint32_t r = 0;
  for (uint32_t k = 0; k < 16; ++k) {
    const int n = int(k & 1u) + int((k >> 1) & 1u) + int((k >> 2) & 1u) + int((k >> 3) & 1u);
    if (mask_mode ? n != 2 : n > 2) r |= 1u << k;
  }
  return r;
}
constexpr uint64_t kPickLut = make_pick_lut();
constexpr uint32_t kFlagMask = make_flag_lut(true);
constexpr uint32_t kFlagExact = make_flag_lut(false);

// Byte lanes whose bit 7 flags "set" -> 4-bit set (bit i = byte i): move the flags to bit
// 0 of each byte and sum the bytes, weighted 1, 2, 4, 8, with one multiply.
__device__ __forceinline__ uint32_t gather_bit7(uint32_t t) {
  return (((t >> 7) & 0x01010101u) * 0x01020408u) >> 24;
}

// Candidate set of one group from its mask word (4 bytes, non-zero = keep): adding 0x7F
// to the low 7 bits of a byte carries into bit 7 unless they are zero.
__device__ __forceinline__ uint32_t keep_from_mask(uint32_t m) {
  return gather_bit7(((m & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | m);
}

// Candidate set of one group from its values: non-zero elements (+0 and -0 are zero for
// the float types).  16-bit: the group is words w0 (elements 0, 1) and w1 (2, 3); the
// same carry trick on 15-bit magnitudes sets bit 15 of each non-zero half.
__device__ __forceinline__ uint32_t keep_nonzero16(uint32_t w0, uint32_t w1) {
  const uint32_t y0 = (w0 & 0x7FFF7FFFu) + 0x7FFF7FFFu, y1 = (w1 & 0x7FFF7FFFu) + 0x7FFF7FFFu;
  return ((y0 >> 15) & 1u) | ((y0 >> 30) & 2u) | ((y1 >> 13) & 4u) | ((y1 >> 28) & 8u);
}
template <int CLS>
__device__ __forceinline__ uint32_t keep_nonzero8(uint32_t w) {
  if constexpr (CLS == kFloat8) return gather_bit7((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu);
  return gather_bit7(((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w);
}

// 4-bit group: four nibbles in the low 16 bits of x.  Non-zero nibbles by the same carry
// trick (bit 3 of each nibble), gathered into a 4-bit set with one multiply.
__device__ __forceinline__ uint32_t keep_nonzero4(uint32_t x) {
  const uint32_t t = ((x & 0x7777u) + 0x7777u) | x;
  return ((((t >> 3) & 0x1111u) * 0x1248u) >> 12) & 0xFu;
}
// The two kept nibbles of a 4-bit group as one byte (p0 low, p1 high).
__device__ __forceinline__ uint32_t pack4(uint32_t x, uint32_t nib) {
  return ((x >> (4 * (nib & 3u))) & 0xFu) | (((x >> (4 * (nib >> 2))) & 0xFu) << 4);
}

// The two kept elements of a 16-bit group (words w0, w1) packed as one word.
__device__ __forceinline__ uint32_t pack16(uint32_t w0, uint32_t w1, uint32_t nib) {
  const uint32_t p0 = nib & 3u, p1 = nib >> 2;
  const uint32_t sel = (p0 * 0x22u + 0x10u) | ((p1 * 0x22u + 0x10u) << 8);
  return __byte_perm(w0, w1, sel);
}
// The two kept bytes of an 8-bit group (word w) in the low 16 bits.
__device__ __forceinline__ uint32_t pack8(uint32_t w, uint32_t nib) {
  return __byte_perm(w, 0u, (nib & 3u) | ((nib >> 2) << 4) | 0x4400u) & 0xFFFFu;
}

// Magnitude mode: keep the two largest |x| of a group; equal magnitudes keep the lower
// position.  Each key k_p (a magnitude below 2^16) becomes the composite (k_p << 2) |
// (3 - p), which orders the positions totally (magnitude first, then lower position), so
// the kept pair is the two largest composites: a four-input max/min network, and the
// positions are the composites' low two bits.  Returns the nibble p0 | p1 << 2.
__device__ __forceinline__ uint32_t top2_keys(uint32_t k0, uint32_t k1, uint32_t k2, uint32_t k3) {
  const uint32_t c0 = (k0 << 2) | 3u, c1 = (k1 << 2) | 2u, c2 = (k2 << 2) | 1u, c3 = k3 << 2;
  const uint32_t a = max(c0, c1), b = min(c0, c1), c = max(c2, c3), d = min(c2, c3);
  const uint32_t t1 = max(a, c);                  // the largest
  const uint32_t t2 = max(min(a, c), max(b, d));  // the second largest
  const uint32_t q1 = ~t1 & 3u, q2 = ~t2 & 3u;    // their positions
  return min(q1, q2) | (max(q1, q2) << 2);
}

// 16-bit group in words w0 (elements 0, 1) and w1 (2, 3); keys = bits without the sign.
__device__ __forceinline__ uint32_t top2_16(uint32_t w0, uint32_t w1) {
  return top2_keys(w0 & 0x7FFFu, (w0 >> 16) & 0x7FFFu, w1 & 0x7FFFu, (w1 >> 16) & 0x7FFFu);
}

// 4-bit group in the low 16 bits: keys = |x| (s4: two's complement, so -8 gives 8).
template <int CLS>
__device__ __forceinline__ uint32_t top2_4(uint32_t x) {
  uint32_t k[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t n = (x >> (4 * p)) & 0xFu;
    if constexpr (CLS == kSigned4) {
      const int v = int(n) - int((n & 8u) << 1);
      k[p] = uint32_t(v < 0 ? -v : v);
    } else {
      k[p] = n;
    }
  }
  return top2_keys(k[0], k[1], k[2], k[3]);
}

// 8-bit group in one word: keys = |x| (FP8: bits without the sign; s8: absolute value,
// so -128 gives 128; u8: the value).
template <int CLS>
__device__ __forceinline__ uint32_t top2_8(uint32_t w) {
  uint32_t k[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint32_t b = (w >> (8 * p)) & 0xFFu;
    if constexpr (CLS == kFloat8) {
      k[p] = b & 0x7Fu;
    } else if constexpr (CLS == kSigned8) {
      const int v = int(b) - int((b & 0x80u) << 1);
      k[p] = uint32_t(v < 0 ? -v : v);
    } else {
      k[p] = b;
    }
  }
  return top2_keys(k[0], k[1], k[2], k[3]);
}

// One 16-byte chunk of a row (8 16-bit, 16 8-bit or 32 4-bit elements = 2, 4 or 8
// groups; EB = element bits): the kept elements packed into 8 bytes, the groups' nibbles
// (4 bits each, group g at 4g) and the mode's rule-break flag in bit 0 of `flags`.
// m: the chunk's mask bytes (mask mode), one word per group.
template <int EB, int CLS, int MODE>
__device__ __forceinline__ void compress_chunk(const uint4& v, const uint32_t (&m)[8], uint2& vals,
                                               uint32_t& nibs, uint32_t& flags) {
  constexpr int kGroups = (128 / EB) / 4;
  constexpr uint32_t kFlags = MODE == 1 ? kFlagMask : kFlagExact;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out[2] = {0, 0};
  nibs = 0;
  flags = 0;
#pragma unroll
  for (int g = 0; g < kGroups; ++g) {
    uint32_t nib;
    uint32_t x4 = 0;  // 4-bit: the group's four nibbles
    if constexpr (EB == 4) x4 = (w[g >> 1] >> (16 * (g & 1))) & 0xFFFFu;
    if constexpr (MODE == 2) {
      if constexpr (EB == 16)
        nib = top2_16(w[2 * g], w[2 * g + 1]);
      else if constexpr (EB == 8)
        nib = top2_8<CLS>(w[g]);
      else
        nib = top2_4<CLS>(x4);
    } else {
      uint32_t keep;
      if constexpr (MODE == 1)
        keep = keep_from_mask(m[g]);
      else if constexpr (EB == 16)
        keep = keep_nonzero16(w[2 * g], w[2 * g + 1]);
      else if constexpr (EB == 8)
        keep = keep_nonzero8<CLS>(w[g]);
      else
        keep = keep_nonzero4(x4);
      nib = uint32_t(kPickLut >> (4 * keep)) & 0xFu;
      flags |= kFlags >> keep;
    }
    if constexpr (EB == 16)
      out[g] = pack16(w[2 * g], w[2 * g + 1], nib);
    else if constexpr (EB == 8)
      out[g >> 1] |= pack8(w[g], nib) << (16 * (g & 1));
    else
      out[g >> 2] |= pack4(x4, nib) << (8 * (g & 3));
    nibs |= nib << (4 * g);
  }
  vals = make_uint2(out[0], out[1]);
}

// One 16-byte chunk of A (row, chunk cc of the row) and, in mask mode, its mask bytes
// (one per element, one word per group).
template <int EB, int MODE>
__device__ __forceinline__ void load_chunk(const CompressArgs& a, int64_t row, int64_t cc,
                                           uint4& v, uint32_t (&m)[8]) {
  constexpr int kElems = 128 / EB;
  v = __ldcs(reinterpret_cast<const uint4*>(a.A + row * a.lda_bytes + cc * 16));
  if constexpr (MODE == 1) {
    if constexpr (kElems == 8) {
      const uint2 mm = __ldcs(reinterpret_cast<const uint2*>(a.mask + row * a.ldm + cc * 8));
      m[0] = mm.x;
      m[1] = mm.y;
    } else {
#pragma unroll
      for (int h = 0; h < kElems / 16; ++h) {  // 16 mask bytes per load
        const uint4 mm = __ldcs(
            reinterpret_cast<const uint4*>(a.mask + row * a.ldm + cc * kElems + 16 * h));
        m[4 * h + 0] = mm.x;
        m[4 * h + 1] = mm.y;
        m[4 * h + 2] = mm.z;
        m[4 * h + 3] = mm.w;
      }
    }
  }
}

// EB = element bits (16, 8 or 4); MODE = SP24_MODE_* value.  Each warp step covers
// kUnroll runs of 32 consecutive chunks; all their loads are issued before any is used,
// so a thread keeps kUnroll 16-byte loads (plus mask loads) in flight.
template <int EB, int CLS, int MODE>
__global__ void __launch_bounds__(256, EB == 4 ? 3 : 4) compress_kernel(CompressArgs a) {
  griddep_launch_dependents();  // the GEMM after this pass may start its prologue
  constexpr int kElems = 128 / EB;   // elements per 16-byte chunk
  constexpr int kGroups = kElems / 4;  // groups per chunk
  constexpr int kLanesPerWord = 32 / kElems;
  constexpr int kUnroll = 4;
  const int lane = threadIdx.x & 31;
  const int64_t cpr = a.K / kElems;  // chunks per row
  const int64_t total = a.M * cpr;
  const bool small = total < (int64_t(1) << 32);  // 32-bit chunk numbers suffice
  const int64_t warp_global = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t warp_stride = (int64_t(gridDim.x) * blockDim.x) >> 5;
  uint32_t any_flag = 0;

  for (int64_t base = warp_global * 32 * kUnroll; base < total;
       base += warp_stride * 32 * kUnroll) {
    uint4 v[kUnroll];
    uint32_t mbits[kUnroll][8];
    int64_t row[kUnroll], cc[kUnroll];
    bool active[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t c = base + u * 32 + lane;
      active[u] = c < total;
      if (small) {
        const uint32_t r = uint32_t(c) / uint32_t(cpr);
        row[u] = r;
        cc[u] = int64_t(uint32_t(c) - r * uint32_t(cpr));
      } else {
        row[u] = c / cpr;
        cc[u] = c - row[u] * cpr;
      }
      v[u] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int q = 0; q < 8; ++q) mbits[u][q] = 0;
      if (active[u]) load_chunk<EB, MODE>(a, row[u], cc[u], v[u], mbits[u]);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      uint2 vals;
      uint32_t nibs, flags;
      compress_chunk<EB, CLS, MODE>(v[u], mbits[u], vals, nibs, flags);
      if (active[u]) any_flag |= flags & 1u;
      if (active[u])
        __stcs(reinterpret_cast<uint2*>(a.values + row[u] * a.ldv_bytes + cc[u] * 8), vals);
      // merge the nibbles of the lanes that share one index word
      uint32_t word = nibs << ((4 * kGroups) * (lane % kLanesPerWord));
      if constexpr (kLanesPerWord > 1) {
#pragma unroll
        for (int o = 1; o < kLanesPerWord; o <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, o);
      }
      if (active[u] && (lane % kLanesPerWord) == 0) {
        a.index[row[u] * a.ldi + (cc[u] * kElems) / 32] = word;
      }
    }
  }
  if (a.status != nullptr && __any_sync(0xFFFFFFFFu, any_flag != 0u) && lane == 0)
    atomicOr(a.status, kDevNot24);
}

// Asynchronous global -> shared copies of one thread (no registers in flight).
__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async8(uint32_t saddr, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(saddr), "l"(g) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Geometry of the fused pass.  A warp's unit is one (16-row band of a 128-row tile, GEMM
// stage): kStageK dense K of 16 rows.  Lane L covers chunk c = L % kCpr of rows
// kRpi * k + L / kCpr (k = 0 .. kIters-1) of the band, so rows r and r + 8 of the band
// sit in the same lane (k and k + kIters / 2).
template <int EB, int MODE, bool kL8>
struct FusedGeo {
  static constexpr int kStageK = kL8 ? 256 : 128;
  static constexpr int kElems = 128 / EB;            // elements per 16-byte chunk
  static constexpr int kCpr = kStageK / kElems;      // chunks per row and stage: 16, 16, 8, 4
  static constexpr int kRpi = 32 / kCpr;             // rows per warp iteration: 2, 2, 4, 8
  static constexpr int kIters = 16 / kRpi;           // 8, 8, 4, 2
  static constexpr int kMaskBytes = MODE == 1 ? kElems : 0;  // mask bytes per chunk
  static constexpr int kUnitBytes = kIters * 32 * (16 + kMaskBytes);  // staged per unit
  // units staged per warp: the one being worked on and kBufs - 1 ahead (mask mode stages
  // more bytes per unit, so fewer fit)
  static constexpr int kBufs = 2;
  static constexpr int kWarps = 4;
  static constexpr int kSmem = kWarps * kBufs * kUnitBytes;
  static_assert(kCpr * kRpi == 32 && kIters * kRpi == 16, "warp tiling");
};

// Compression and the sparse GEMM's metadata image in one pass (the image the separate
// re-layout kernel in meta.cu writes from the canonical index; its layout is described
// there).  Each warp compresses its unit's 16 rows over the stage's K range chunk by chunk
// as compress_kernel does (values and canonical index words, which stay the interchange
// format; index may be null), then writes the band's 16 TMEM lanes of the stage's image
// block with 16-byte stores (the words of a lane gathered by shuffles).  Rows beyond M and
// K beyond the operand count as all-zero groups (pattern {0,1}): the image padding.
// kL8: the FP8 layout (256 dense K per stage, lane = row, the row's 8 canonical words);
// otherwise the 16-bit layout (128 dense K per stage; lane 16b + l of band b holds 16-bit
// halves h = l/8 of the canonical words of rows l%8 and l%8 + 8), also used by integers.
//
// Loads: every lane copies the chunks (and mask bytes) it will use into its warp's
// shared-memory ring with cp.async, two units ahead of the one it works on, so each SM
// keeps 2 x (warps) units of A in flight without holding them in registers.  A lane only
// ever reads back what it copied itself, so its own cp.async.wait_group is the only
// synchronisation (no barrier, no spin).
template <int EB, int CLS, int MODE, bool kL8>
__global__ void __launch_bounds__(128) compress_meta_kernel(CompressArgs a) {
  griddep_launch_dependents();  // the GEMM after this pass may start its prologue
  using G = FusedGeo<EB, MODE, kL8>;
  constexpr int kElems = G::kElems, kCpr = G::kCpr, kRpi = G::kRpi, kIters = G::kIters;
  constexpr int kGroups = kElems / 4;
  constexpr int kLanesPerWord = kElems < 32 ? 32 / kElems : 1;
  constexpr int kHalves = kElems >= 16 ? kElems / 16 : 1;  // 16-K halves a chunk starts
  constexpr uint32_t kPadWord = 0x44444444u;
  constexpr uint32_t kPadNibs = kGroups == 8 ? kPadWord : (kPadWord >> (32 - 4 * kGroups));
  constexpr int kLaneVecs = kL8 ? 2 : 1;  // 16-byte vectors per TMEM lane in an image block
  static_assert(!kL8 || EB == 8, "the FP8 layout holds 8-bit elements");
  extern __shared__ __align__(16) uint8_t fused_smem[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = lane % kCpr, rsub = lane / kCpr;
  const int64_t units = a.mtiles * 8 * a.ksteps;
  const int64_t warp0 = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  uint4* meta = reinterpret_cast<uint4*>(a.meta);
  uint8_t* ring = fused_smem + warp * (G::kBufs * G::kUnitBytes);
  uint32_t any_flag = 0;

  // rows of the band (from row0 = first row of this lane) that exist, capped
  auto rows_left = [&](int64_t row0) -> int {
    const int64_t r = a.M - row0;
    return r > 16 ? 16 : int(r);
  };
  const int64_t a_step = kRpi * a.lda_bytes, m_step = kRpi * a.ldm;
  const int64_t v_step = kRpi * a.ldv_bytes, i_step = kRpi * a.ldi;

  // stage unit u into ring buffer `buf` (always commits a group, possibly empty)
  auto issue = [&](int64_t u, int buf) {
    if (u < units) {
      const int64_t band = u / a.ksteps, s = u - band * a.ksteps;
      const int64_t cc = s * kCpr + c;
      const int64_t row0 = band * 16 + rsub;
      const int left = rows_left(row0);
      const uint32_t sb = smem_addr(ring + buf * G::kUnitBytes);
      if (cc * kElems < a.K) {
        const uint8_t* ag = a.A + row0 * a.lda_bytes + cc * 16;
        const uint8_t* mg = MODE == 1 ? a.mask + row0 * a.ldm + cc * kElems : nullptr;
#pragma unroll
        for (int k = 0; k < kIters; ++k) {
          if (kRpi * k < left) {
            cp_async16(sb + (k * 32 + lane) * 16, ag);
            if constexpr (MODE == 1) {
              const uint32_t ms = sb + kIters * 32 * 16 + (k * 32 + lane) * G::kMaskBytes;
              if constexpr (kElems == 8) {
                cp_async8(ms, mg);
              } else {
#pragma unroll
                for (int h = 0; h < kElems / 16; ++h) cp_async16(ms + 16 * h, mg + 16 * h);
              }
            }
          }
          ag += a_step;
          if constexpr (MODE == 1) mg += m_step;
        }
      }
    }
    cp_async_commit();
  };

#pragma unroll
  for (int b = 0; b < G::kBufs - 1; ++b) issue(warp0 + b * nwarps, b);
  int buf = 0;
  for (int64_t u = warp0; u < units; u += nwarps) {
    issue(u + (G::kBufs - 1) * nwarps, buf == 0 ? G::kBufs - 1 : buf - 1);
    cp_async_wait<G::kBufs - 1>();  // this lane's copies of unit u have landed
    const int64_t band = u / a.ksteps, s = u - band * a.ksteps;
    const int64_t cc = s * kCpr + c;              // chunk of the row
    const bool kin = cc * kElems < a.K;
    const int64_t row0 = band * 16 + rsub;
    const int left = rows_left(row0);
    uint8_t* vg = a.values + row0 * a.ldv_bytes + cc * 8;
    uint32_t* ig = a.index + row0 * a.ldi + (cc * kElems) / 32;
    const uint8_t* st = ring + buf * G::kUnitBytes;
    // the band's lanes of the (tile, stage) block: the block starts at uint4
    // (tile * ksteps + s) * kLaneVecs * 128, lane L at + L * kLaneVecs, the band at lane
    // (band % 8) * 16
    uint4* img = meta + ((band >> 3) * a.ksteps + s) * (kLaneVecs * 128) + (band & 7) * 16 * kLaneVecs;
    uint32_t half16[kIters][kHalves];
#pragma unroll
    for (int k = 0; k < kIters; ++k) {
      const bool valid = kin && kRpi * k < left;
      uint4 v = make_uint4(0, 0, 0, 0);
      uint32_t m[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (valid) {
        v = *reinterpret_cast<const uint4*>(st + (k * 32 + lane) * 16);
        if constexpr (MODE == 1) {
          const uint8_t* ms = st + kIters * 32 * 16 + (k * 32 + lane) * G::kMaskBytes;
          if constexpr (kElems == 8) {
            const uint2 mm = *reinterpret_cast<const uint2*>(ms);
            m[0] = mm.x;
            m[1] = mm.y;
          } else {
#pragma unroll
            for (int h = 0; h < kElems / 16; ++h) {
              const uint4 mm = *reinterpret_cast<const uint4*>(ms + 16 * h);
              m[4 * h + 0] = mm.x;
              m[4 * h + 1] = mm.y;
              m[4 * h + 2] = mm.z;
              m[4 * h + 3] = mm.w;
            }
          }
        }
      }
      uint2 vals;
      uint32_t nibs, flags;
      compress_chunk<EB, CLS, MODE>(v, m, vals, nibs, flags);
      if (!valid) nibs = kPadNibs;
      if (valid) {
        any_flag |= flags & 1u;
        __stcs(reinterpret_cast<uint2*>(vg), vals);
      }
      vg += v_step;
      // the row's canonical word of this chunk, merged across the lanes that share it
      uint32_t word = nibs << ((4 * kGroups) * (lane % kLanesPerWord));
      if constexpr (kLanesPerWord > 1) {
#pragma unroll
        for (int o = 1; o < kLanesPerWord; o <<= 1) word |= __shfl_xor_sync(0xFFFFFFFFu, word, o);
      }
      if (valid && a.index != nullptr && (lane % kLanesPerWord) == 0) *ig = word;
      ig += i_step;
      if constexpr (kL8) {
        // the row's lane takes its 8 canonical words of the stage in order (MMA j reads
        // words 2j and 2j + 1); lane c holds word c / 2, so lanes c = 0 and c = 8 gather
        // words 0-3 and 4-7 and write them
        const uint32_t w1 = __shfl_xor_sync(0xFFFFFFFFu, word, 2);
        const uint32_t w2 = __shfl_xor_sync(0xFFFFFFFFu, word, 4);
        const uint32_t w3 = __shfl_xor_sync(0xFFFFFFFFu, word, 6);
        if ((c & 7) == 0) img[(kRpi * k + rsub) * 2 + (c >> 3)] = make_uint4(word, w1, w2, w3);
      } else {
#pragma unroll
        for (int i = 0; i < kHalves; ++i) {
          const int hidx = (c * kElems) / 16 + i;  // 16-K half of the stage (0 .. 7)
          half16[k][i] = (word >> (16 * (hidx & 1))) & 0xFFFFu;
        }
      }
    }
    if constexpr (!kL8) {
      // TMEM lane r + 8h of the band (r < 8) takes, for MMA j, 16-K half 2j + h of rows r
      // (low 16 bits) and r + 8 (high).  Half hidx of a row is held by the lane of chunk
      // (hidx / kHalves) * kChunksPerHalf, as its value i = hidx % kHalves; the lane of
      // chunk h gathers the four words of lane r + 8h and writes its 16 bytes.
      constexpr int kChunksPerHalf = kElems >= 16 ? 1 : 16 / kElems;
#pragma unroll
      for (int k = 0; k < kIters / 2; ++k) {
        uint32_t wv[kHalves];
#pragma unroll
        for (int i = 0; i < kHalves; ++i) wv[i] = half16[k][i] | (half16[k + kIters / 2][i] << 16);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t w[kMmasPerStage];
#pragma unroll
          for (int j = 0; j < kMmasPerStage; ++j) {
            const int hidx = 2 * j + h;
            const int cs = (hidx / kHalves) * kChunksPerHalf;
            w[j] = __shfl_sync(0xFFFFFFFFu, wv[hidx % kHalves], rsub * kCpr + cs);
          }
          if (c == h) img[kRpi * k + rsub + 8 * h] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
    buf = buf == G::kBufs - 1 ? 0 : buf + 1;
  }
  cp_async_wait<0>();
  if (a.status != nullptr && __any_sync(0xFFFFFFFFu, any_flag != 0u) && lane == 0)
    atomicOr(a.status, kDevNot24);
}

// expand(values, index): one thread writes one 16-byte chunk of dense A.
template <int EB>
__global__ void __launch_bounds__(256) decompress_kernel(DecompressArgs a) {
  constexpr int kElems = 128 / EB;
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
      if constexpr (EB == 16) {
        k0 = kv[g] & 0xFFFFu;
        k1 = kv[g] >> 16;
      } else if constexpr (EB == 8) {
        const uint32_t h = (kv[g >> 1] >> (16 * (g & 1))) & 0xFFFFu;
        k0 = h & 0xFFu;
        k1 = h >> 8;
      } else {
        const uint32_t b = (kv[g >> 2] >> (8 * (g & 3))) & 0xFFu;
        k0 = b & 0xFu;
        k1 = b >> 4;
      }
      // element 4g + p gets k0 at p0, k1 at p1, zero elsewhere (static register indices)
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint32_t v = uint32_t(p) == p0 ? k0 : (uint32_t(p) == p1 ? k1 : 0u);
        const int e = 4 * g + p;
        if constexpr (EB == 16)
          o[e >> 1] |= v << (16 * (e & 1));
        else if constexpr (EB == 8)
          o[e >> 2] |= v << (8 * (e & 3));
        else
          o[e >> 3] |= v << (4 * (e & 7));
      }
    }
    *reinterpret_cast<uint4*>(a.A + row * a.lda_bytes + cc * 16) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

template <int EB, int CLS>
cudaError_t launch_compress_cls(const CompressArgs& a, int mode, int grid, cudaStream_t s) {
  switch (mode) {
    case 0: compress_kernel<EB, CLS, 0><<<grid, 256, 0, s>>>(a); break;
    case 1: compress_kernel<EB, CLS, 1><<<grid, 256, 0, s>>>(a); break;
    default: compress_kernel<EB, CLS, 2><<<grid, 256, 0, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, int dtype, int mode, int num_sms,
                            cudaStream_t s) {
  const int64_t chunks = a.M * (a.K / (128 / elem_bits(dtype)));
  // each thread covers 4 chunks per step; 8 resident blocks of 256 threads per SM
  int64_t want = (chunks + 1023) / 1024;
  int64_t cap = int64_t(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
  switch (dtype) {
    case kF16:
    case kBF16: return launch_compress_cls<16, kFloat16>(a, mode, grid, s);
    case kE4M3:
    case kE5M2: return launch_compress_cls<8, kFloat8>(a, mode, grid, s);
    case kS8: return launch_compress_cls<8, kSigned8>(a, mode, grid, s);
    case kU8: return launch_compress_cls<8, kUnsigned8>(a, mode, grid, s);
    case kS4: return launch_compress_cls<4, kSigned4>(a, mode, grid, s);
    default: return launch_compress_cls<4, kUnsigned4>(a, mode, grid, s);
  }
}

namespace {
// Blocks of 4 warps; as many per SM as the shared-memory rings allow (queried once per
// kernel instance).
template <int EB, int CLS, int MODE, bool kL8>
cudaError_t launch_compress_meta_mode(const CompressArgs& a, int num_sms, cudaStream_t s) {
  using G = FusedGeo<EB, MODE, kL8>;
  static int per_sm = 0;  // 0: not yet set up
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (per_sm == 0) {
      auto k = compress_meta_kernel<EB, CLS, MODE, kL8>;
      if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem) !=
              cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, G::kWarps * 32, G::kSmem) !=
              cudaSuccess ||
          per_sm < 1) {
        per_sm = 0;
        return cudaErrorInvalidConfiguration;
      }
    }
  }
  const int64_t units = a.mtiles * 8 * a.ksteps;  // one warp per (band, stage) at a time
  int64_t want = (units + G::kWarps - 1) / G::kWarps;
  int64_t cap = int64_t(num_sms) * per_sm;
  const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
  compress_meta_kernel<EB, CLS, MODE, kL8><<<grid, G::kWarps * 32, G::kSmem, s>>>(a);
  return cudaGetLastError();
}

template <int EB, int CLS, bool kL8>
cudaError_t launch_compress_meta_cls(const CompressArgs& a, int mode, int num_sms,
                                     cudaStream_t s) {
  switch (mode) {
    case 0: return launch_compress_meta_mode<EB, CLS, 0, kL8>(a, num_sms, s);
    case 1: return launch_compress_meta_mode<EB, CLS, 1, kL8>(a, num_sms, s);
    default: return launch_compress_meta_mode<EB, CLS, 2, kL8>(a, num_sms, s);
  }
}
}  // namespace

cudaError_t launch_compress_meta(const CompressArgs& a, int dtype, int mode, int num_sms,
                                 cudaStream_t s) {
  switch (dtype) {
    case kF16:
    case kBF16: return launch_compress_meta_cls<16, kFloat16, false>(a, mode, num_sms, s);
    case kE4M3:
    case kE5M2: return launch_compress_meta_cls<8, kFloat8, true>(a, mode, num_sms, s);
    case kS8: return launch_compress_meta_cls<8, kSigned8, false>(a, mode, num_sms, s);
    case kU8: return launch_compress_meta_cls<8, kUnsigned8, false>(a, mode, num_sms, s);
    case kS4: return launch_compress_meta_cls<4, kSigned4, false>(a, mode, num_sms, s);
    default: return launch_compress_meta_cls<4, kUnsigned4, false>(a, mode, num_sms, s);
  }
}

cudaError_t launch_decompress(const DecompressArgs& a, int dtype, int num_sms, cudaStream_t s) {
  const int eb = elem_bits(dtype);
  const int64_t chunks = a.M * (a.K / (128 / eb));
  int64_t want = (chunks + 255) / 256;
  int64_t cap = int64_t(num_sms) * 8;
  const int grid = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
  if (eb == 16)
    decompress_kernel<16><<<grid, 256, 0, s>>>(a);
  else if (eb == 8)
    decompress_kernel<8><<<grid, 256, 0, s>>>(a);
  else
    decompress_kernel<4><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace sp24
