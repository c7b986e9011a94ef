// spmma.cu -- the 2:4 sparse GEMM D = expand(A_c, meta) * B + C on sm_103a tensor cores.
//
// Semantics: "RDNA4 sparse WMMA builtins", "Builtin reference" (each builtin returns
// expand(srcA, index) x srcB + srcC, f32 accumulate); "v_smfmac_f32_32x32x32_bf8_bf8",
// "Semantics" (D = A(sparse) * B + D).  The pages' kernels issue one 16x16 (or 32x32)
// builtin per wavefront per K step from LDS tiles; here one elected thread issues
// tcgen05.mma.sp on whole 128- or 256-row tiles whose accumulators live in tensor memory.
//
// Variants of one kernel:
//   pair    (N > 128):  a cluster of two CTAs per 256 x 256 tile, cta_group::2: each CTA
//           stages its own 128 rows of A and its own 128-column half of B and the even
//           CTA issues the MMAs, so each loaded byte feeds twice the work.  The 256-column
//           accumulator is single-buffered; eight epilogue warps drain it to registers
//           first and release it before they add C and store.  With 16-bit float
//           operands, when the last round of tiles would leave more than half of the CTA
//           pairs idle, those tiles run as two 256 x 128 halves each.
//           Integer products (widened to bf16) use it too, summing f32 chunks into int32.
//   pair 256 x 128 (16-bit operands with 32 < N <= 128): the same with 64-column halves
//           of B and 256-K stages (see Geo).
//   single  (FP8 with 32 < N <= 128): one CTA per 128 x 128 tile, cta_group::1,
//           accumulator double-buffered in TMEM so the epilogue of one tile overlaps the
//           next.
//   narrow  (N <= 32): one CTA per 128 x 32 tile (see Geo).
// Warp roles (persistent over tiles, one CTA per SM):
//   warp 0   TMA producer: per stage one box of compressed A (K-major, 128-byte swizzle)
//            and the B boxes (K x N row-major = MN-major, 128-byte swizzle).
//   warp 1   TMEM owner and MMA issuer: per stage 4 x tcgen05.mma.sp and one
//            tcgen05.commit that frees the stage.
//   warps 4+ epilogue: tcgen05.ld, + C, cast to f32 / bf16, 16-byte stores.
//   last 4   metadata writers, one per quarter of the TMEM lanes: each lane's words of a
//            stage (16 bytes, FP8 32, of the image block) are loaded from global memory a
//            few stages ahead and stored into the MMAs' 16-column-aligned TMEM slots (slot
//            set = ring stage) by tcgen05.st.  Measured on the GB300 with operands resident in
//            shared memory, a tcgen05.cp of the metadata in front of every MMA costs the
//            tensor pipe about 44 cycles per MMA (bf16 M=128, N=256: 204 cycles against
//            160), stores from other warps nothing measurable.
// Every mbarrier wait is bounded; a wait that gives up sets SP24_DEV_TIMEOUT in the
// caller's status word and the CTA drains its in-flight work and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "../../include/sp24.h"
#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {
namespace {

constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = 128 * 128;  // one stage of compressed A: 128 rows x 128 bytes
constexpr int kSlotCols = 16;       // TMEM columns per MMA metadata slot (aligned)
constexpr uint32_t kPadWord = 0x44444444u;  // pattern {0,1} in every group: rows / K past A
// Integer mode: integers widened to bf16 are exact, and the f32 accumulator holds an exact
// integer as long as every partial sum stays within 2^24.  A chunk of MmaParams::chunk
// stages (128 dense K each, half of them kept products) is sized for that: s8 x s8
// (|a b| <= 2^14): 2048 dense K, 1024 products; u8 x s8 (|a b| <= 255 * 128): 1024 dense K;
// 4-bit (|a b| <= 225): 8192 dense K.  The epilogue adds the chunks in int32
// (two's-complement wrap).

struct MmaParams {
  const void* C;
  void* D;
  int64_t ldc, ldd;
  int32_t* status;
  int c32, d32;  // C / D rows allow 32-byte vector accesses (base and pitch 32-byte aligned)
  int ctype;     // float C: 0 = f32, 1 = bf16, 2 = f16
  int chunk;     // integer mode: stages per exactly-summed f32 chunk
  int d_f16;     // 16-bit float D (OUT == 1): 0 = bf16, 1 = f16
  int batoms;    // B boxes loaded per stage and CTA (the narrow variant skips empty ones)
  int M, N, K;
  int mtiles, ntiles, num_kb;  // tiles of the variant (128 or 256 rows, 128 or 256 cols)
  int img_kb;                  // metadata image stages per 128-row tile (a stage of the
                               // narrow and 256 x 128 16-bit variants spans two)
  int band_rows;               // tile order: bands of this many rows of D, swept along N
  int batch;                   // problems of equal shape; problem b's C / D start at
  int64_t stride_c, stride_d;  // C + b * stride_c, D + b * stride_d (elements)
  const uint8_t* meta;         // metadata image; problem b's at meta + b * stride_meta
  int64_t stride_meta;         // (bytes)
  const uint32_t* index;       // or, for one problem, the canonical index itself (M x K/32
  int64_t ldi;                 // words, pitch ldi); then meta is unused
  int idx_vec;                 // index base 16-byte aligned and ldi % 4 == 0: 16-byte loads
  uint64_t limit_ns;
  int units;            // work units of the launch: tiles, plus the split tiles' halves
  int n_full;           // units below n_full are whole tiles; the rest are halves (N / 2)
  uint32_t idesc_half;  // instruction descriptor of a half tile
  int diag_stall;  // self-test: the TMA producer issues nothing, so every wait gives up
};

// Variants: pair (256 x 256 tiles on a CTA pair; also the integer path), pair with
// 256 x 128 tiles and double-buffered accumulators (16-bit operands with 32 < N <= 128),
// single (128 x 128 tiles: FP8 with 32 < N <= 128) and narrow (128 x 32 tiles for
// N <= 32: B staged in 32-byte swizzle atoms, so a stage holds only the columns that
// exist).  The narrow and 256 x 128 products move little data per MMA, so their stages
// are as long as the MMA thread's and the metadata writers' fixed cost per stage allows to
// hide: 16-bit operands take two image stages (256 dense K, 8 MMAs, two boxes of A) per
// stage, and three such stages fill the TMEM columns left for metadata slots (the 256 x 128
// tiles then keep a single 128-column accumulator: measured faster than two accumulators
// with 128-K stages, also on shapes with many tiles per CTA pair).
template <int ESZ, bool kPair, bool kNarrow = false, bool kHalfN = false>
struct Geo {
  static constexpr int kImgStageK = ESZ == 2 ? 128 : 256;    // dense K per image stage
  static constexpr int kImgPer = ((kNarrow || kHalfN) && ESZ == 2) ? 2 : 1;  // per stage
  static constexpr int kStageK = kImgStageK * kImgPer;        // dense K per stage
  static constexpr int kMmaK = ESZ == 2 ? 32 : 64;            // dense K per MMA
  static constexpr int kMmas = kStageK / kMmaK;               // 4 (narrow 16-bit: 8)
  static constexpr int kImgWords = ESZ == 1 ? 8 : 4;          // per TMEM lane, image stage
  static constexpr int kImgBytes = 128 * 4 * kImgWords;       // image block: 2 / 4 KB
  static constexpr int kMetaWords = kImgPer * kImgWords;      // per TMEM lane and stage
  static constexpr int kABoxes = kImgPer;                     // 128 x 128-byte A boxes
  static constexpr int kAStage = kABoxes * kABytes;           // compressed A per stage
  static constexpr int kTileM = kPair ? 256 : 128;
  static constexpr int kTileN = kPair ? (kHalfN ? 128 : 256) : (kNarrow ? 32 : 128);
  static constexpr int kBCols = kPair ? kTileN / 2 : kTileN;  // B columns staged per CTA
  static constexpr int kAtomInner = kNarrow ? 32 : 128;       // bytes of a B atom row
  static constexpr int kSwzCode = kNarrow ? 6 : 2;            // descriptor: 32B / 128B
  static constexpr int kAtomN = kAtomInner / ESZ;             // B columns per atom
  static constexpr int kAtoms = kBCols / kAtomN;
  static constexpr int kAtomBytes = kStageK * kAtomInner;     // one B box
  static constexpr int kBBytes = kAtoms * kAtomBytes;
  static constexpr int kStages = kImgPer == 2 ? 3 : (kNarrow ? 7 : 4);
  static constexpr int kStageBytes = kAStage + kBBytes;  // the metadata skips shared memory
  // CTA pairs: one 4 KiB staging box per epilogue warp (32 rows x 32 f32 columns) through
  // which the epilogue's C tiles arrive and its D tiles leave by TMA
  static constexpr int kStgBytes = kPair ? 8 * 4096 : 0;
  static constexpr int kSmemBytes = kStages * kStageBytes + kStgBytes + 1024;
  static constexpr int kAccBufs = (kPair && (!kHalfN || kImgPer == 2)) ? 1 : 2;
  static constexpr int kAccCols = kAccBufs * kTileN;
  static constexpr uint32_t kMetaCol = kAccCols;              // slot set s at + s * 64
  // warps: 0 TMA producer, 1 MMA issuer, 2-3 idle, then the epilogue warps, then four
  // metadata writers (warp id % 4 = the TMEM lane quarter each may access)
  static constexpr int kEpiWarps = kPair ? 8 : 4;
  static constexpr int kEpiWarp0 = 4;
  static constexpr int kWriterWarp0 = kEpiWarp0 + kEpiWarps;
  static constexpr int kThreads = 32 * (kWriterWarp0 + 4);    // 512 or 384
  // pair: 512 threads launch with 128 registers each; the producer / MMA warpgroup and
  // the writer warpgroup give theirs down to kRegsLight so the two epilogue warpgroups
  // can hold the drained accumulator (kRegsEpi); the shares add up to at most the launch's
  static constexpr uint32_t kRegsLight = 56;
  static constexpr uint32_t kRegsEpi = 200;
  static_assert(!kPair || (kRegsLight * 256 + kRegsEpi * 256 <= 65536u), "register split");
  static_assert(kAccCols + kStages * kMmas * kSlotCols <= int(kTmemCols), "TMEM budget");
  static_assert(kSmemBytes <= 232448 - 512, "shared memory budget");
  // one CTA per SM: a product launched early behind another (programmatic dependent
  // launch) never shares an SM, and so its TMEM, with a CTA of the one before it
  static_assert(2 * kSmemBytes > 232448, "one CTA per SM");
  static_assert(kAtoms >= 1, "B atoms");
};

// Tile order: bands of MmaParams::band_rows rows of D, each swept along N, so that the
// tiles in flight at one time (about one per CTA pair) share a few row blocks of A and
// column blocks of B that stay in L2 instead of streaming all of A for every column of
// tiles.  Taller bands re-read B from DRAM fewer times; measured on the GB300: 4096-row
// bands for N >= 4096 (FP8 8192^3 3% faster than 2048), 2048 otherwise (LLM N = 2048 2%
// faster than 4096).
inline int band_rows_for(int64_t N) { return N >= 4096 ? 4096 : 2048; }
template <int kTileM>
__device__ __forceinline__ void tile_coords(const MmaParams& p, int t, int& mt, int& nt);

// Tile t of the whole launch: problem b = t / (tiles of one problem), then the tile's
// (row tile, column tile) inside it.
template <int kTileM>
__device__ __forceinline__ void batch_tile(const MmaParams& p, int t, int& b, int& mt, int& nt) {
  const int per = p.mtiles * p.ntiles;
  b = t / per;
  tile_coords<kTileM>(p, t - b * per, mt, nt);
}

template <int kTileM>
__device__ __forceinline__ void tile_coords(const MmaParams& p, int t, int& mt, int& nt) {
  const int kBand = p.band_rows / kTileM;  // row tiles per band
  const int band_tiles = kBand * p.ntiles;
  const int g = t / band_tiles, r = t - g * band_tiles;
  const int rest = p.mtiles - g * kBand;
  const int gm = rest < kBand ? rest : kBand;  // the last band may be shorter
  mt = g * kBand + r % gm;
  nt = r / gm;
}

// Quad transpose (the four threads t with equal t/4 exchange values): thread q = t%4
// holds, for j = 0..3, the two values at columns 8j + 2q and +1 of a 32-column row
// segment in v[2j], v[2j+1]; afterwards it holds columns 8q .. 8q+7 in v[0..7].  Two
// butterfly stages (partners q^1, then q^2), each swapping the two elements whose index
// bit differs from the thread's.
__device__ __forceinline__ void quad_transpose(float (&v)[8], int q) {
#pragma unroll
  for (int bit = 1; bit <= 2; bit <<= 1) {
    const bool up = (q & bit) != 0;
#pragma unroll
    for (int j0 = 0; j0 < 4; ++j0) {
      if (j0 & bit) continue;
      const int j1 = j0 | bit;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float send = up ? v[2 * j0 + c] : v[2 * j1 + c];
        const float recv = __shfl_xor_sync(0xFFFFFFFFu, send, bit);
        if (up)
          v[2 * j0 + c] = recv;
        else
          v[2 * j1 + c] = recv;
      }
    }
  }
}

__device__ __forceinline__ void ld_f32x8(const float* src, bool v32, float (&c)[8]) {
  if (v32) {
    asm volatile("ld.global.cs.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3]), "=f"(c[4]), "=f"(c[5]),
                   "=f"(c[6]), "=f"(c[7])
                 : "l"(src));
  } else {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(src));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(src) + 1);
    c[0] = a.x; c[1] = a.y; c[2] = a.z; c[3] = a.w;
    c[4] = b.x; c[5] = b.y; c[6] = b.z; c[7] = b.w;
  }
}

// one 16-bit float (bf16 if !f16) as f32: exact
__device__ __forceinline__ float half_bits_to_f32(uint32_t h, bool f16) {
  return f16 ? __half2float(__ushort_as_half(static_cast<unsigned short>(h)))
             : __uint_as_float(h << 16);
}

// C at 8 consecutive columns of one output row, as f32 (C is f32, bf16 or f16 by
// p.ctype); zeros beyond M, N or without C.
__device__ __forceinline__ void load_c8(float (&c)[8], const MmaParams& p, int row, int col,
                                        int64_t cofs) {
  if (p.C == nullptr || row >= p.M || col >= p.N) {
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = 0.f;
    return;
  }
  if (p.ctype == 0) {
    const float* crow = static_cast<const float*>(p.C) + cofs + int64_t(row) * p.ldc + col;
    if (col + 8 <= p.N) {
      ld_f32x8(crow, p.c32 != 0, c);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) c[j] = col + j < p.N ? crow[j] : 0.f;
    }
    return;
  }
  const bool f16 = p.ctype == 2;
  const uint16_t* crow = static_cast<const uint16_t*>(p.C) + cofs + int64_t(row) * p.ldc + col;
  if (col + 8 <= p.N) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(crow));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c[2 * j] = half_bits_to_f32(w[j] & 0xFFFFu, f16);
      c[2 * j + 1] = half_bits_to_f32(w[j] >> 16, f16);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) c[j] = col + j < p.N ? half_bits_to_f32(crow[j], f16) : 0.f;
  }
}

// Cast and store 8 consecutive columns of one output row; columns at or beyond N are not
// touched.  Each quad of threads covers one 32-column segment of a row, so a warp's
// store is 8 whole 128-byte lines (f32 output).
template <int OUT>
__device__ __forceinline__ void store8(const float (&v)[8], const MmaParams& p, int row, int col,
                                       int64_t dofs) {
  if (row >= p.M || col >= p.N) return;
  const bool full = col + 8 <= p.N;
  if constexpr (OUT == 0) {
    float* d = static_cast<float*>(p.D) + dofs + int64_t(row) * p.ldd + col;
    if (full) {
      if (p.d32) {
        asm volatile("st.global.cs.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(d), "f"(v[0]),
                     "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                     : "memory");
      } else {
        __stcs(reinterpret_cast<float4*>(d), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(d) + 1, make_float4(v[4], v[5], v[6], v[7]));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col + j < p.N) d[j] = v[j];
    }
  } else if (p.d_f16) {
    __half* d = static_cast<__half*>(p.D) + dofs + int64_t(row) * p.ldd + col;
    if (full) {
      __half2 h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
      uint4 u;
      memcpy(&u, h, 16);
      __stcs(reinterpret_cast<uint4*>(d), u);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col + j < p.N) d[j] = __float2half_rn(v[j]);
    }
  } else {
    __nv_bfloat16* d = static_cast<__nv_bfloat16*>(p.D) + dofs + int64_t(row) * p.ldd + col;
    if (full) {
      __nv_bfloat162 h[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      uint4 u;
      memcpy(&u, h, 16);
      __stcs(reinterpret_cast<uint4*>(d), u);
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (col + j < p.N) d[j] = __float2bfloat16_rn(v[j]);
    }
  }
}

// kSeg 32-column segments (columns col0 .. col0 + 32 kSeg - 1) of one output row from a
// .16x256b fragment r (repetitions 0 .. 4 kSeg - 1; row half e = 0 is lane t/4, e = 1
// lane t/4 + 8): up to two segments at a time, their C loads issued together, then each
// segment is transposed across the quad, added to C and stored.
template <int OUT, int kSeg>
__device__ __forceinline__ void store_row(const uint32_t* r, int e, const MmaParams& p, int row,
                                          int col0, int q, int64_t cofs, int64_t dofs) {
  constexpr int kBatch = kSeg < 2 ? kSeg : 2;
#pragma unroll
  for (int g0 = 0; g0 < kSeg; g0 += kBatch) {
    float c[kBatch][8];
#pragma unroll
    for (int g = 0; g < kBatch; ++g) load_c8(c[g], p, row, col0 + 32 * (g0 + g) + 8 * q, cofs);
#pragma unroll
    for (int g = 0; g < kBatch; ++g) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = p.K > 0 ? __uint_as_float(r[4 * (4 * (g0 + g) + j) + 2 * e]) : 0.f;
        v[2 * j + 1] = p.K > 0 ? __uint_as_float(r[4 * (4 * (g0 + g) + j) + 2 * e + 1]) : 0.f;
      }
      quad_transpose(v, q);
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] += c[g][j];
      store8<OUT>(v, p, row, col0 + 32 * (g0 + g) + 8 * q, dofs);
    }
  }
}

// Pull this thread's share of the C rows of a coming tile into L2 (the quad leader of
// each row, one bulk prefetch of up to `cols` columns per row).
__device__ __forceinline__ void prefetch_c_rows(const MmaParams& p, int row0, int col0, int q,
                                                int cols, int64_t cofs) {
  if (p.C == nullptr || q != 0 || col0 >= p.N) return;
  const int ncols = p.N - col0 < cols ? p.N - col0 : cols;
  const int csize = p.ctype == 0 ? 4 : 2;
  const uint32_t bytes = uint32_t(ncols * csize) & ~15u;
  if (bytes == 0) return;
#pragma unroll
  for (int h = 0; h < 2; ++h)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int row = row0 + 16 * h + 8 * e;
      if (row < p.M)
        bulk_prefetch_l2(static_cast<const uint8_t*>(p.C) +
                             (cofs + int64_t(row) * p.ldc + col0) * csize,
                         bytes);
    }
}

// 32 consecutive columns of one output row held by one thread (a 32x32b accumulator
// load): add C, cast and store as 8-column pieces (32-byte f32 / 16-byte 16-bit vectors).
template <int OUT>
__device__ __forceinline__ void store_row32(const uint32_t (&r)[32], const MmaParams& p, int row,
                                            int col0, int64_t cofs, int64_t dofs) {
  float c[4][8];
#pragma unroll
  for (int g = 0; g < 4; ++g) load_c8(c[g], p, row, col0 + 8 * g, cofs);
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    float v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (p.K > 0 ? __uint_as_float(r[8 * g + j]) : 0.f) + c[g][j];
    store8<OUT>(v, p, row, col0 + 8 * g, dofs);
  }
}

// Byte offset of 16-byte piece j of row r inside a TMA box whose rows are kRowBytes long
// (128: SWIZZLE_128B, 64: SWIZZLE_64B): the piece index is XOR-ed with address bits 7+.
template <int kRowBytes>
__device__ __forceinline__ uint32_t stg_offset(int r, int j) {
  constexpr uint32_t kMask = kRowBytes == 128 ? 7u : 3u;
  const uint32_t off = uint32_t(r * kRowBytes + j * 16);
  return off ^ (((off >> 7) & kMask) << 4);
}

// Epilogue of one 32-column chunk of one 32-row block through a staging box in shared
// memory: the thread of row `lane` adds its row of C (already in the box, in C's type)
// to the accumulator values v and writes the row of D (in D's type) over it.
template <int OUT>
__device__ __forceinline__ void stage_chunk(uint8_t* stg, int lane, float (&v)[32], bool hasC,
                                            int ctype, bool d_f16) {
  if (hasC) {
    if (ctype == 0) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 c = *reinterpret_cast<const float4*>(stg + stg_offset<128>(lane, j));
        v[4 * j] += c.x;
        v[4 * j + 1] += c.y;
        v[4 * j + 2] += c.z;
        v[4 * j + 3] += c.w;
      }
    } else {
      const bool f16 = ctype == 2;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 u = *reinterpret_cast<const uint4*>(stg + stg_offset<64>(lane, j));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          v[8 * j + 2 * k] += half_bits_to_f32(w[k] & 0xFFFFu, f16);
          v[8 * j + 2 * k + 1] += half_bits_to_f32(w[k] >> 16, f16);
        }
      }
    }
  }
  if constexpr (OUT == 0) {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4*>(stg + stg_offset<128>(lane, j)) =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float a = v[8 * j + 2 * k], b = v[8 * j + 2 * k + 1];
        if (d_f16) {
          const __half2 h = __floats2half2_rn(a, b);
          memcpy(&w[k], &h, 4);
        } else {
          const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
          memcpy(&w[k], &h, 4);
        }
      }
      *reinterpret_cast<uint4*>(stg + stg_offset<64>(lane, j)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
  }
}

// Integer epilogue for one 32-column chunk: D = sum + C (s32, nullable), wrapping.
__device__ __forceinline__ void store_chunk_s32(const uint32_t* v, const MmaParams& p, int row,
                                                int col0) {
  uint32_t o[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) o[j] = v[j];
  const bool full = col0 + 32 <= p.N;
  if (p.C != nullptr) {
    const int32_t* crow = static_cast<const int32_t*>(p.C) + int64_t(row) * p.ldc + col0;
    if (full) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const int4 cv = __ldcs(reinterpret_cast<const int4*>(crow + j));
        o[j] += uint32_t(cv.x);
        o[j + 1] += uint32_t(cv.y);
        o[j + 2] += uint32_t(cv.z);
        o[j + 3] += uint32_t(cv.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < p.N) o[j] += uint32_t(crow[j]);
    }
  }
  int32_t* drow = static_cast<int32_t*>(p.D) + int64_t(row) * p.ldd + col0;
  if (full) {
#pragma unroll
    for (int j = 0; j < 32; j += 4)
      __stcs(reinterpret_cast<int4*>(drow + j),
             make_int4(int(o[j]), int(o[j + 1]), int(o[j + 2]), int(o[j + 3])));
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (col0 + j < p.N) drow[j] = int32_t(o[j]);
  }
}

// A grouped launch: up to kMaxGroup problems of different shapes (same element types)
// whose tiles share one persistent grid.  Everything the kernel reads per problem, tensor
// maps included, travels in kernel parameter space (about 11 KB), so the launch needs no
// device memory of its own.
constexpr int kMaxGroup = 32;
static_assert(kMaxGroup == kMaxGroupPerLaunch, "one group table per launch");
struct GroupTable {
  CUtensorMap a[kMaxGroup], b[kMaxGroup];
  const uint8_t* meta[kMaxGroup];
  int count;
  int tile_start[kMaxGroup + 1];  // problem g owns launch tiles tile_start[g] .. [g+1]-1
  int M[kMaxGroup], N[kMaxGroup], K[kMaxGroup], num_kb[kMaxGroup], img_kb[kMaxGroup];
  int mtiles[kMaxGroup], ntiles[kMaxGroup], batoms[kMaxGroup];
  uint32_t idesc[kMaxGroup];
  const void* C[kMaxGroup];
  void* D[kMaxGroup];
  int64_t ldc[kMaxGroup], ldd[kMaxGroup];
  int c32[kMaxGroup], d32[kMaxGroup];
};

// The problem a launch tile belongs to (0 without a group table) and its tile number
// inside that problem.
template <bool kGrouped>
__device__ __forceinline__ int tile_problem(const GroupTable* gt, int t, int& local) {
  if constexpr (!kGrouped) {
    local = t;
    return 0;
  } else {
    int g = 0;
    while (g + 1 < gt->count && t >= gt->tile_start[g + 1]) ++g;
    local = t - gt->tile_start[g];
    return g;
  }
}

// Unit u of a one-problem launch: the whole tile u below n_full; above, the halves of
// the remaining tiles (half 0: the tile's first kTileN / 2 columns, half 1: the rest).
__device__ __forceinline__ void unit_tile(const MmaParams& p, int u, int& t, int& hf) {
  if (u < p.n_full) {
    t = u;
    hf = -1;
  } else {
    const int h = u - p.n_full;
    t = p.n_full + (h >> 1);
    hf = h & 1;
  }
}

// The kernel parameters as one problem of a group sees them (the launch's own parameters
// without a group table).
template <bool kGrouped>
__device__ __forceinline__ void problem_params(const MmaParams& p, const GroupTable* gt, int g,
                                               MmaParams& q) {
  if constexpr (kGrouped) {
    q = p;
    q.M = gt->M[g];
    q.N = gt->N[g];
    q.K = gt->K[g];
    q.num_kb = gt->num_kb[g];
    q.img_kb = gt->img_kb[g];
    q.mtiles = gt->mtiles[g];
    q.ntiles = gt->ntiles[g];
    q.batoms = gt->batoms[g];
    q.C = gt->C[g];
    q.D = gt->D[g];
    q.ldc = gt->ldc[g];
    q.ldd = gt->ldd[g];
    q.c32 = gt->c32[g];
    q.d32 = gt->d32[g];
    q.batch = 1;
    q.stride_c = q.stride_d = 0;
    q.meta = gt->meta[g];
    q.stride_meta = 0;
  } else {
    (void)p, (void)gt, (void)g, (void)q;
  }
}

// OUT: 0 = f32 output, 1 = 16-bit float output (bf16 or f16 by p.d_f16), 2 = s32 output
// (integer mode).  C (nullable) is f32, bf16 or f16 (p.ctype) for float outputs, s32 for
// integer mode.
// kGrouped: the tiles of the problems of a group table (tmA/tmB/idesc unused);
// otherwise one problem, or a strided batch, with tensor maps tmA, tmB.
template <int ESZ, int OUT, bool kPair, bool kNarrow, bool kHalfN, bool kGrouped>
__device__ __forceinline__ void spmma_body(const CUtensorMap* tmA, const CUtensorMap* tmB,
                                           const CUtensorMap* tmC, const CUtensorMap* tmD,
                                           const MmaParams& p,
                                           const uint32_t idesc, const GroupTable* gt) {
  using G = Geo<ESZ, kPair, kNarrow, kHalfN>;
  constexpr int kStages = G::kStages;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  // full_bar (even CTA): the stage's operands of both CTAs have landed (TMA bytes) and every
  // metadata writer warp of the pair has stored the stage's metadata into its TMEM slots
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], drain_bar;
  __shared__ __align__(8) uint64_t stg_bar[8];  // CTA pairs: a C tile has reached a staging box
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;
  const int unit = kPair ? int(blockIdx.x >> 1) : int(blockIdx.x);
  const int nunits = kPair ? int(gridDim.x >> 1) : int(gridDim.x);
  uint8_t* sA = smem;
  uint8_t* sB = sA + kStages * G::kAStage;
  uint8_t* sStg = sB + kStages * G::kBBytes;  // 1024-byte aligned (stage sizes are)
  const int ntiles_total = kGrouped ? gt->tile_start[gt->count] : p.units;
  // CTA pairs with 16-bit float operands may split the tiles of the last, partial round
  // into halves (host decision: n_full < units)
  constexpr bool kHalves = kPair && !kHalfN && !kGrouped && ESZ == 2 && OUT != 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1 + 4 * (kPair ? 2 : 1));  // producer + writer warps
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], G::kEpiWarps * (kPair ? 2 : 1));
    }
    mbar_init(&drain_bar, 1);
    for (int w = 0; w < 8; ++w) mbar_init(&stg_bar[w], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if constexpr (!kGrouped) {
      prefetch_tmap(tmA);
      prefetch_tmap(tmB);
    }
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(&tmem_slot, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&tmem_slot, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();  // the peer's barriers exist before any remote use
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  volatile int* abort = &abort_flag;
  // Programmatic dependent launch: the prologue above may overlap the kernel before this
  // one on the stream, and the next product on the stream may start its own prologue on
  // SMs this grid leaves free or frees (a CTA of it cannot share an SM with one of this
  // grid: each takes more than half of the shared memory).  Every role that touches
  // global memory first waits (griddep_wait) until the kernel before has completed and its
  // writes are visible; the MMA thread touches none.
  griddep_launch_dependents();

  // Roles by warpgroup (the pair variant re-divides the register file per warpgroup, so
  // each role's code sits under its warpgroup's setmaxnreg)
  if (warp < G::kEpiWarp0) {
    if constexpr (kPair) regs_dec<G::kRegsLight>();
  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0 && !p.diag_stall && unit < ntiles_total) {
      // While the kernel before may still run, pull this CTA's first stages into L2.  L2
      // is where every write of that kernel lands, so a line fetched early is updated by
      // those writes; the loads below read it only after the wait.
      int lt, hf = -1;
      const int g = tile_problem<kGrouped>(gt, unit, lt);
      if constexpr (kHalves) unit_tile(p, unit, lt, hf);
      MmaParams qg;
      problem_params<kGrouped>(p, gt, g, qg);
      const MmaParams& pp = kGrouped ? qg : p;
      const CUtensorMap* mA = kGrouped ? &gt->a[g] : tmA;
      const CUtensorMap* mB = kGrouped ? &gt->b[g] : tmB;
      int b, mt, nt;
      batch_tile<G::kTileM>(pp, lt, b, mt, nt);
      const int mt128 = kPair ? mt * 2 + int(rank) : mt;
      const int bcol = hf < 0 ? nt * G::kTileN + int(rank) * G::kBCols
                              : nt * G::kTileN + hf * (G::kTileN / 2) + int(rank) * (G::kBCols / 2);
      const int na = hf < 0 ? pp.batoms : G::kAtoms / 2;
      for (int kb = 0; kb < pp.num_kb && kb < kStages; ++kb) {
        const int kx = kb * (G::kStageK / 2);
        for (int i = 0; i < G::kABoxes; ++i)
          if (2 * (kx + i * (128 / ESZ)) < pp.K) tma_prefetch_3d(mA, kx + i * (128 / ESZ), mt128 * 128, b);
        for (int a = 0; a < G::kAtoms; ++a)
          if (a < na) tma_prefetch_3d(mB, bcol + a * G::kAtomN, kb * G::kStageK, b);
      }
    }
    griddep_wait();
    if (lane == 0 && !p.diag_stall) {
      int q = 0;
      for (int t = unit; t < ntiles_total && !*abort; t += nunits) {
        int lt, hf = -1;
        const int g = tile_problem<kGrouped>(gt, t, lt);
        if constexpr (kHalves) unit_tile(p, t, lt, hf);
        MmaParams qg;
        problem_params<kGrouped>(p, gt, g, qg);
        const MmaParams& pp = kGrouped ? qg : p;
        const CUtensorMap* mA = kGrouped ? &gt->a[g] : tmA;
        const CUtensorMap* mB = kGrouped ? &gt->b[g] : tmB;
        int b, mt, nt;
        batch_tile<G::kTileM>(pp, lt, b, mt, nt);
        const int mt128 = kPair ? mt * 2 + int(rank) : mt;  // this CTA's 128-row tile
        // a half tile: each CTA stages half of its usual B columns (one atom)
        const int bcol = hf < 0 ? nt * G::kTileN + int(rank) * G::kBCols
                                : nt * G::kTileN + hf * (G::kTileN / 2) + int(rank) * (G::kBCols / 2);
        const int na = hf < 0 ? pp.batoms : G::kAtoms / 2;
        const uint32_t btx = uint32_t(na * G::kAtomBytes);
        for (int kb = 0; kb < pp.num_kb; ++kb, ++q) {
          const int s = q % kStages;
          if (!mbar_wait(&empty_bar[s], ((q / kStages) & 1) ^ 1u, abort, p.limit_ns)) break;
          const int kx = kb * (G::kStageK / 2);  // compressed elements
          // boxes of A that hold any K (the last stage of a ragged K may need fewer)
          int nbox = 1;
          if constexpr (G::kABoxes > 1)
            while (nbox < G::kABoxes && 2 * (kx + nbox * (128 / ESZ)) < pp.K) ++nbox;
          if (rank == 0)
            mbar_arrive_expect_tx(&full_bar[s],
                                  (uint32_t(nbox * kABytes) + btx) * (kPair ? 2u : 1u));
          if constexpr (kPair) {
            const uint32_t fb = mapa(&full_bar[s], 0);
            for (int i = 0; i < nbox; ++i)
              tma_load_3d_pair(sA + s * G::kAStage + i * kABytes, mA, fb, kx + i * (128 / ESZ),
                               mt128 * 128, b);
#pragma unroll
            for (int a = 0; a < G::kAtoms; ++a)
              if (a < na)
                tma_load_3d_pair(sB + s * G::kBBytes + a * G::kAtomBytes, mB, fb,
                                 bcol + a * G::kAtomN, kb * G::kStageK, b);
          } else {
            for (int i = 0; i < nbox; ++i)
              tma_load_3d(sA + s * G::kAStage + i * kABytes, mA, &full_bar[s],
                          kx + i * (128 / ESZ), mt128 * 128, b);
#pragma unroll
            for (int a = 0; a < G::kAtoms; ++a)
              if (a < pp.batoms)
                tma_load_3d(sB + s * G::kBBytes + a * G::kAtomBytes, mB, &full_bar[s],
                            bcol + a * G::kAtomN, kb * G::kStageK, b);
          }
        }
      }
      if (*abort) {  // give copies already issued time to land before the CTA exits
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (rank == 0 && lane == 0) {
      const uint64_t adesc_hi = smem_desc_hi(16, 1024, 2);
      // B is MN-major: LBO = next atom along N, SBO = next 8 rows of K
      const uint64_t bdesc_hi = smem_desc_hi(G::kAtomBytes, 8 * G::kAtomInner, G::kSwzCode);
      int q = 0, local = 0, chunk = 0;
      bool ready = false;  // stage q's full_bar phase is known to have completed
      for (int t = unit; t < ntiles_total && !*abort; t += nunits, ++local) {
        int lt, hf = -1;
        const int g = tile_problem<kGrouped>(gt, t, lt);
        if constexpr (kHalves) unit_tile(p, t, lt, hf);
        const int num_kb = kGrouped ? gt->num_kb[g] : p.num_kb;
        const int kdense = kGrouped ? gt->K[g] : p.K;
        const uint32_t id = kGrouped ? gt->idesc[g] : (hf < 0 ? idesc : p.idesc_half);
        bool ok = true;
        int abuf = 0;
        uint32_t d_tmem = tmem;
        if constexpr (OUT != 2) {
          abuf = G::kAccBufs == 1 ? 0 : (local & 1);
          const int use = G::kAccBufs == 1 ? local : (local >> 1);  // earlier uses of abuf
          if (!mbar_wait(&acc_empty[abuf], (use & 1) ^ 1u, abort, p.limit_ns)) break;
          tc_fence_after();
          d_tmem = tmem + uint32_t(abuf * G::kTileN);
        }
        int kc = 0;  // stage within an integer chunk (kb % p.chunk, counted)
        for (int kb = 0; kb < num_kb; ++kb, ++q, kc = (kc + 1 == p.chunk) ? 0 : kc + 1) {
          const int s = q % kStages;
          const uint32_t par = (q / kStages) & 1;
          if constexpr (OUT == 2) {
            if (kc == 0) {  // new chunk: next accumulator buffer
              abuf = G::kAccBufs == 1 ? 0 : (chunk & 1);
              const int cuse = G::kAccBufs == 1 ? chunk : (chunk >> 1);  // earlier uses
              if (!mbar_wait(&acc_empty[abuf], (cuse & 1) ^ 1u, abort, p.limit_ns)) {
                ok = false;
                break;
              }
              tc_fence_after();
              d_tmem = tmem + uint32_t(abuf * G::kTileN);
            }
          }
          // the stage's operands (both CTAs) and its metadata in the TMEM slots (the writer
          // warps of both CTAs arrive on the same barrier); skipped when the previous
          // stage's test already saw the phase complete
          if (!ready && !mbar_wait(&full_bar[s], par, abort, p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t e_tmem = tmem + G::kMetaCol + uint32_t(s * G::kMmas * kSlotCols);
          const uint32_t a_saddr = smem_addr(sA + s * G::kAStage);
          const uint32_t b_saddr = smem_addr(sB + s * G::kBBytes);
          const int k0 = kb * G::kStageK;
          const int first = (OUT == 2) ? kc : kb;  // accumulate unless the chunk/tile starts
          if (k0 + G::kStageK <= kdense) {
            // the whole stage in one sequence, testing the next stage's barrier meanwhile
            // (MMA j: A 32 bytes further along K, B kMmaK rows further, metadata slot j)
            const int qn = q + 1;
            if constexpr (G::kMmas == 8)  // 256-K stages: two boxes of A, 8 MMAs
              ready = mma_stage8_test_next<kPair>(
                  smem_addr(&full_bar[qn % kStages]), uint32_t((qn / kStages) & 1), d_tmem,
                  smem_desc(a_saddr, adesc_hi), smem_desc(b_saddr, bdesc_hi), 32u / 16u,
                  uint32_t(kABytes / 16), uint32_t(G::kMmaK * G::kAtomInner / 16), e_tmem, id,
                  first > 0 ? 1u : 0u, smem_addr(&empty_bar[s]));
            else
              ready = mma_stage_test_next<kPair, ESZ == 1>(
                  smem_addr(&full_bar[qn % kStages]), uint32_t((qn / kStages) & 1), d_tmem,
                  smem_desc(a_saddr, adesc_hi), smem_desc(b_saddr, bdesc_hi), 32u / 16u,
                  uint32_t(G::kMmaK * G::kAtomInner / 16), e_tmem, id, first > 0 ? 1u : 0u,
                  smem_addr(&empty_bar[s]));
          } else {  // the last, partial stage of a ragged K
            ready = false;
#pragma unroll
            for (int j = 0; j < G::kMmas; ++j) {
              if (k0 + j * G::kMmaK < kdense) {
                const uint64_t ad = smem_desc(a_saddr + (j / 4) * kABytes + 32 * (j % 4), adesc_hi);
                const uint64_t bd = smem_desc(b_saddr + j * G::kMmaK * G::kAtomInner, bdesc_hi);
                const uint32_t acc = (first > 0 || j > 0) ? 1u : 0u;
                if constexpr (kPair)
                  tc_mma_sp_pair<ESZ == 1>(d_tmem, ad, bd, e_tmem + j * kSlotCols, id, acc);
                else
                  tc_mma_sp<ESZ == 1>(d_tmem, ad, bd, e_tmem + j * kSlotCols, id, acc);
              }
            }
            if constexpr (kPair)
              tc_commit_pair_mc(&empty_bar[s], 3);
            else
              tc_commit(&empty_bar[s]);
          }
          if constexpr (OUT == 2) {
            if (kc == p.chunk - 1 || kb == num_kb - 1) {  // chunk done
              if constexpr (kPair)
                tc_commit_pair_mc(&acc_full[abuf], 3);
              else
                tc_commit(&acc_full[abuf]);
              ++chunk;
            }
          }
        }
        if (!ok) break;
        if constexpr (OUT != 2) {
          if constexpr (kPair)
            tc_commit_pair_mc(&acc_full[abuf], 3);
          else
            tc_commit(&acc_full[abuf]);
        }
      }
      // every MMA issued by this thread completes before TMEM can be released
      if constexpr (kPair)
        tc_commit_pair(&drain_bar);
      else
        tc_commit(&drain_bar);
      mbar_wait_drain(&drain_bar, 0, 1000000000ull);
    }
  }  // warps 2 and 3 have no role
  } else if (warp >= G::kWriterWarp0) {
    if constexpr (kPair) regs_dec<G::kRegsLight>();
    // ---------------------------------------------------------------- metadata writers
    // Warp w stores TMEM lanes 32 (w % 4) .. +31 of each stage's four metadata slots.  A
    // lane's words for a stage are loaded from global memory a few stages early into
    // registers: 16 (FP8: 32) bytes of the image block, or, reading the canonical index
    // directly, the canonical words they are made of (16-bit layout: 4 words of each of the
    // lane's two rows, combined by halves at store time; FP8: the row's 8 words).  Once the
    // MMAs that last read the slot set are done (empty_bar, the producer's barrier) the
    // warp stores them with tcgen05.st, waits for the stores and arrives on the even CTA's
    // full_bar of the stage, which the MMA issuer waits on before the stage's MMAs.
    const int quad = warp & 3;
    const int lrow = quad * 32 + lane;            // this thread's TMEM lane
    // kind::f16 layout: TMEM lane 16b + l holds halves h = l / 8 of rows 16b + l % 8 and
    // 16b + l % 8 + 8 of the tile
    const int h16 = (lrow >> 3) & 1;
    const int r16 = (lrow & ~15) + (lrow & 7);
    const uint32_t full_addr = kPair ? mapa(&full_bar[0], 0) : smem_addr(&full_bar[0]);
    const uint32_t lanes = tmem + (uint32_t(quad * 32) << 16) + G::kMetaCol;
    // a cursor over this CTA's stages in the producer's order: tile t, stage kb of num_kb,
    // the tile's first row and the address of this lane's image words of that stage
    struct Cursor {
      int t, kb, num_kb, img_kb, row0;
      const uint4* src;
    };
    auto seek = [&](Cursor& c, int t) {  // first stage of tile t or a later one
      for (c.t = t; c.t < ntiles_total; c.t += nunits) {
        int lt, hf = -1;
        const int g = tile_problem<kGrouped>(gt, c.t, lt);
        if constexpr (kHalves) unit_tile(p, c.t, lt, hf);
        (void)hf;
        MmaParams qg;
        problem_params<kGrouped>(p, gt, g, qg);
        const MmaParams& pp = kGrouped ? qg : p;
        if (pp.num_kb == 0) continue;
        int b, mt, nt;
        batch_tile<G::kTileM>(pp, lt, b, mt, nt);
        const int mt128 = kPair ? mt * 2 + int(rank) : mt;
        c.kb = 0;
        c.num_kb = pp.num_kb;
        c.img_kb = pp.img_kb;
        c.row0 = mt128 * 128;
        c.src = pp.meta == nullptr
                    ? nullptr
                    : reinterpret_cast<const uint4*>(pp.meta + b * pp.stride_meta +
                                                     int64_t(mt128) * pp.img_kb * G::kImgBytes) +
                          lrow * (G::kImgWords / 4);
        return;
      }
    };
    auto next = [&](Cursor& c) {
      if (c.src != nullptr) c.src += G::kImgPer * G::kImgBytes / 16;
      if (++c.kb == c.num_kb) seek(c, c.t + nunits);
    };
    auto writers = [&](auto index_mode) {
      constexpr bool kIdx = decltype(index_mode)::value;
      constexpr int kAhead = kIdx ? 2 : 4;         // stages of words held in registers
      // words per lane and stage: the image's, or the canonical words they are made of
      // (16-bit: one word per MMA of each of the lane's two rows; FP8: two words per MMA of
      // the lane's row)
      constexpr int kW = kIdx ? 2 * G::kMmas : G::kMetaWords;
      auto load = [&](const Cursor& c, uint32_t (&w)[kW]) {
        if (c.t >= ntiles_total) return;
        if constexpr (kIdx) {
          const int kw = p.K / 32;  // canonical words per row
          if constexpr (ESZ == 2) {
            constexpr int kR = G::kMmas;  // words of each row in the stage
            const int ra = c.row0 + r16;
            if (p.idx_vec && c.kb * kR + kR <= kw && ra + 8 < p.M) {
              // the stage's words of each row are contiguous 16-byte vectors
              const uint4* lo = reinterpret_cast<const uint4*>(p.index + int64_t(ra) * p.ldi + c.kb * kR);
              const uint4* hi = reinterpret_cast<const uint4*>(p.index + int64_t(ra + 8) * p.ldi + c.kb * kR);
#pragma unroll
              for (int v = 0; v < kR / 4; ++v) {
                const uint4 x = __ldg(lo + v), y = __ldg(hi + v);
                w[4 * v] = x.x, w[4 * v + 1] = x.y, w[4 * v + 2] = x.z, w[4 * v + 3] = x.w;
                w[kR + 4 * v] = y.x, w[kR + 4 * v + 1] = y.y, w[kR + 4 * v + 2] = y.z,
                           w[kR + 4 * v + 3] = y.w;
              }
              return;
            }
#pragma unroll
            for (int j = 0; j < kR; ++j) {
              const int col = c.kb * kR + j;
              w[j] = (col < kw && ra < p.M) ? __ldg(p.index + int64_t(ra) * p.ldi + col) : kPadWord;
              w[kR + j] = (col < kw && ra + 8 < p.M)
                              ? __ldg(p.index + int64_t(ra + 8) * p.ldi + col)
                              : kPadWord;
            }
          } else {
            const int r = c.row0 + lrow;
            if (p.idx_vec && c.kb * kW + kW <= kw && r < p.M) {
              // the stage's words of the row are contiguous 16-byte vectors
              const uint4* src = reinterpret_cast<const uint4*>(p.index + int64_t(r) * p.ldi + c.kb * kW);
#pragma unroll
              for (int v = 0; v < kW / 4; ++v) {
                const uint4 x = __ldg(src + v);
                w[4 * v] = x.x, w[4 * v + 1] = x.y, w[4 * v + 2] = x.z, w[4 * v + 3] = x.w;
              }
              return;
            }
#pragma unroll
            for (int i = 0; i < kW; ++i) {
              const int col = c.kb * kW + i;
              w[i] = (col < kw && r < p.M) ? __ldg(p.index + int64_t(r) * p.ldi + col) : kPadWord;
            }
          }
        } else {
          // the lane's words of each image stage the kernel stage covers (past the last
          // image stage of a ragged K: the pad pattern)
#pragma unroll
          for (int i = 0; i < G::kImgPer; ++i) {
            const bool in = c.kb * G::kImgPer + i < c.img_kb;
#pragma unroll
            for (int v = 0; v < G::kImgWords / 4; ++v) {
              const uint4 x = in ? __ldg(c.src + i * (G::kImgBytes / 16) + v)
                                 : make_uint4(kPadWord, kPadWord, kPadWord, kPadWord);
              uint32_t* o = w + i * G::kImgWords + 4 * v;
              o[0] = x.x;
              o[1] = x.y;
              o[2] = x.z;
              o[3] = x.w;
            }
          }
        }
      };
      Cursor ld, wr;
      seek(ld, unit);
      wr = ld;
      if constexpr (!kIdx) {
        // the first stages' image blocks of the first tile into L2 before the wait (see
        // the producer)
        if (quad == 0 && lane == 0 && ld.t < ntiles_total) {
          const int n = ld.img_kb < kStages * G::kImgPer ? ld.img_kb : kStages * G::kImgPer;
          bulk_prefetch_l2(ld.src - lrow * (G::kImgWords / 4), uint32_t(n * G::kImgBytes));
        }
      }
      griddep_wait();
      uint32_t buf[kAhead][kW];
#pragma unroll
      for (int a = 0; a < kAhead; ++a) {
        load(ld, buf[a]);
        if (ld.t < ntiles_total) next(ld);
      }
      int q = 0;
      bool ok = true;
      while (ok && wr.t < ntiles_total) {
#pragma unroll
        for (int a = 0; a < kAhead; ++a) {
          if (wr.t >= ntiles_total) break;
          const int s = q % kStages;
          int free_slot = 1;
          if (lane == 0)
            free_slot = mbar_wait(&empty_bar[s], ((q / kStages) & 1) ^ 1u, abort, p.limit_ns);
          if (__shfl_sync(0xFFFFFFFFu, free_slot, 0) == 0) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t e = lanes + uint32_t(s * G::kMmas * kSlotCols);
          if constexpr (ESZ == 2) {  // kind::f16: one column per MMA
#pragma unroll
            for (int j = 0; j < G::kMmas; ++j) {
              uint32_t x = buf[a][j];
              if constexpr (kIdx)
                x = ((buf[a][j] >> (16 * h16)) & 0xFFFFu) |
                    (((buf[a][G::kMmas + j] >> (16 * h16)) & 0xFFFFu) << 16);
              tc_st_32x32b_x1(e + j * kSlotCols, x);
            }
          } else {  // kind::f8f6f4: two columns per MMA
#pragma unroll
            for (int j = 0; j < G::kMmas; ++j)
              tc_st_32x32b_x2(e + j * kSlotCols, buf[a][2 * j], buf[a][2 * j + 1]);
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kPair)
              mbar_arrive_cluster(full_addr + uint32_t(s * sizeof(uint64_t)));
            else
              mbar_arrive(&full_bar[s]);
          }
          // refill this register slot with the stage kAhead further on
          load(ld, buf[a]);
          if (ld.t < ntiles_total) next(ld);
          next(wr);
          ++q;
        }
      }
    };
    if (p.index != nullptr)
      writers(std::true_type{});
    else
      writers(std::false_type{});
  } else {
    if constexpr (kPair) regs_inc<G::kRegsEpi>();
    // ---------------------------------------------------------------- epilogue
    griddep_wait();  // C is read and D written only after the kernel before has completed
    const int ew = warp - G::kEpiWarp0;
    const int quad = warp & 3;  // TMEM lanes 32*quad .. +31 (hardware rule: warp id % 4)
    const uint32_t acc_empty_addr =
        kPair ? mapa(&acc_empty[0], 0) : smem_addr(&acc_empty[0]);
    int local = 0, ichunk = 0;
    uint32_t stg_phase = 0;  // C tiles this warp has loaded into its staging box
    for (int t = unit; t < ntiles_total; t += nunits, ++local) {
      int lt, hf = -1;
      const int g = tile_problem<kGrouped>(gt, t, lt);
      if constexpr (kHalves) unit_tile(p, t, lt, hf);
      MmaParams qg;
      problem_params<kGrouped>(p, gt, g, qg);
      const MmaParams& pp = kGrouped ? qg : p;
      int b, mt, nt;
      batch_tile<G::kTileM>(pp, lt, b, mt, nt);
      const int64_t cofs = b * pp.stride_c, dofs = b * pp.stride_d;

      const int abuf = G::kAccBufs == 1 ? 0 : (local & 1);
      const int use = G::kAccBufs == 1 ? local : (local >> 1);
      if constexpr (OUT != 2) {
        if (!mbar_wait(&acc_full[abuf], use & 1, abort, pp.limit_ns)) break;
        tc_fence_after();
      }
      const int row = mt * G::kTileM + int(rank) * 128 + quad * 32 + lane;
      const uint32_t lane_base = tmem + (uint32_t(quad * 32) << 16) + uint32_t(abuf * G::kTileN);
      if constexpr (OUT == 2) {
        // integer mode: one f32 chunk per pp.chunk stages, summed exactly in int32; each
        // thread owns one row x kIntCols columns (pair 256 x 256: 128)
        (void)abuf;
        constexpr int kIntCols = G::kTileN * 4 / G::kEpiWarps;
        const int cbase = (ew >> 2) * kIntCols;  // this warp's first column in the tile
        uint32_t sum[kIntCols];
#pragma unroll
        for (int j = 0; j < kIntCols; ++j) sum[j] = 0u;
        const int nch = (pp.num_kb + pp.chunk - 1) / pp.chunk;
        bool ok = true;
        for (int c = 0; c < nch; ++c, ++ichunk) {
          const int b = G::kAccBufs == 1 ? 0 : (ichunk & 1);
          const int cuse = G::kAccBufs == 1 ? ichunk : (ichunk >> 1);
          if (!mbar_wait(&acc_full[b], cuse & 1, abort, pp.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t base =
              tmem + (uint32_t(quad * 32) << 16) + uint32_t(b * G::kTileN + cbase);
#pragma unroll
          for (int q4 = 0; q4 < kIntCols / 32; ++q4) {
            uint32_t r[32];
            tc_ld_32x32b_x32(base + uint32_t(q4 * 32), r);
            tc_wait_ld();
            if (q4 == kIntCols / 32 - 1) {
              // the whole chunk is in registers: free the accumulator before the last adds
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(acc_empty_addr + uint32_t(b * sizeof(uint64_t)));
            }
#pragma unroll
            for (int j = 0; j < 32; ++j)
              sum[q4 * 32 + j] += uint32_t(__float2int_rn(__uint_as_float(r[j])));
          }
        }
        if (!ok) break;
        if (tmD != nullptr) {
          // C (s32) in and D (s32) out by TMA through this warp's staging box, as the
          // float epilogue does
          uint8_t* stg = sStg + ew * 4096;
          const int row0w = mt * G::kTileM + int(rank) * 128 + quad * 32;
          const bool hasC = pp.C != nullptr;
#pragma unroll
          for (int c = 0; c < kIntCols / 32; ++c) {
            const int col = nt * G::kTileN + cbase + c * 32;
            if (col >= pp.N || row0w >= pp.M) break;
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
            if (hasC) {
              if (lane == 0) {
                mbar_arrive_expect_tx(&stg_bar[ew], 32u * 32u * 4u);
                tma_load_3d(stg, tmC, &stg_bar[ew], col, row0w, 0);
              }
              if (!mbar_wait(&stg_bar[ew], stg_phase & 1u, abort, pp.limit_ns)) {
                mbar_wait_drain(&stg_bar[ew], stg_phase & 1u, 2000000ull);
                ok = false;
                break;
              }
              ++stg_phase;
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              uint4* piece = reinterpret_cast<uint4*>(stg + stg_offset<128>(lane, j));
              uint4 o = make_uint4(sum[c * 32 + 4 * j], sum[c * 32 + 4 * j + 1],
                                   sum[c * 32 + 4 * j + 2], sum[c * 32 + 4 * j + 3]);
              if (hasC) {  // two's-complement wrap
                const uint4 cv = *piece;
                o.x += cv.x;
                o.y += cv.y;
                o.z += cv.z;
                o.w += cv.w;
              }
              *piece = o;
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(tmD, stg, col, row0w, 0);
              bulk_commit_group();
            }
          }
          if (!ok) break;
        } else if (row < pp.M) {
#pragma unroll
          for (int c = 0; c < kIntCols / 32; ++c) {
            const int col0 = nt * G::kTileN + cbase + c * 32;
            if (col0 < pp.N) store_chunk_s32(&sum[c * 32], pp, row, col0);
          }
        }
      } else if constexpr (kPair) {
        // drain this warp's 32 rows x kCols columns (its half of the CTA's columns) with
        // 32x32b loads, one row per thread, free the accumulator, then add C and store
        // each thread's row as 32-byte pieces.  Unlike a transposed layout this takes no
        // shuffles: the epilogue's instructions share issue slots with the MMA thread.
        constexpr int kCols = G::kTileN / 2;  // 128 (256 x 256 tiles) or 64 (256 x 128)
        constexpr int kChunks = kCols / 32;
        const int half = ew >> 2;
        // a half tile (N / 2 columns) gives each warp half as many columns
        const int cols = hf < 0 ? kCols : kCols / 2;
        const int nch = cols / 32;
        uint32_t r[kChunks][32];
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          if (c < nch) tc_ld_32x32b_x32(lane_base + uint32_t(half * cols + 32 * c), r[c]);
        tc_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_addr + uint32_t(abuf * sizeof(uint64_t)));
        const int row = mt * G::kTileM + int(rank) * 128 + quad * 32 + lane;
        const int col0 = nt * G::kTileN + (hf < 0 ? 0 : hf * (G::kTileN / 2)) + half * cols;
        // C is not pulled into L2 ahead of time: a tile's worth prefetched one main loop
        // early was partly evicted again before its use (measured on bf16 4096^3 with f32 C:
        // 176 instead of 134 MB read from DRAM per launch, and 5% slower)
        if (tmD != nullptr) {
          // through this warp's staging box: C arrives by TMA, D leaves by TMA (rows and
          // columns past M and N are zero-filled on the way in and not written on the way out)
          uint8_t* stg = sStg + ew * 4096;
          const int row0w = mt * G::kTileM + int(rank) * 128 + quad * 32;
          const bool hasC = pp.C != nullptr;
          const uint32_t cbytes = 32u * 32u * (pp.ctype == 0 ? 4u : 2u);
          bool ok = true;
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            const int col = col0 + 32 * c;
            if (c >= nch || col >= pp.N || row0w >= pp.M) break;
            if (lane == 0) bulk_wait_read_all();  // the box's previous D has left
            __syncwarp();
            if (hasC) {
              if (lane == 0) {
                mbar_arrive_expect_tx(&stg_bar[ew], cbytes);
                tma_load_3d(stg, tmC, &stg_bar[ew], col, row0w, b);
              }
              if (!mbar_wait(&stg_bar[ew], stg_phase & 1u, abort, pp.limit_ns)) {
                // giving up: let the copy already issued land before the CTA ends
                mbar_wait_drain(&stg_bar[ew], stg_phase & 1u, 2000000ull);
                ok = false;
                break;
              }
              ++stg_phase;
            }
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = pp.K > 0 ? __uint_as_float(r[c][j]) : 0.f;
            stage_chunk<OUT>(stg, lane, v, hasC, pp.ctype, pp.d_f16 != 0);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(tmD, stg, col, row0w, b);
              bulk_commit_group();
            }
          }
          if (!ok) break;
        } else if (row < pp.M) {
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            if (c < nch && col0 + 32 * c < pp.N)
              store_row32<OUT>(r[c], pp, row, col0 + 32 * c, cofs, dofs);
        }
      } else {
        const int row0 = mt * G::kTileM + quad * 32 + (lane >> 2);
        if (t + nunits < ntiles_total) {  // the next tile's C, needed one mainloop from now
          int b2, mt2, nt2;
          int lt2;
          const int g2 = tile_problem<kGrouped>(gt, t + nunits, lt2);
          MmaParams qg2;
          problem_params<kGrouped>(p, gt, g2, qg2);
          const MmaParams& pp2 = kGrouped ? qg2 : p;
          batch_tile<G::kTileM>(pp2, lt2, b2, mt2, nt2);
          prefetch_c_rows(pp2, mt2 * G::kTileM + quad * 32 + (lane >> 2), nt2 * G::kTileN,
                          lane & 3, G::kTileN, b2 * pp2.stride_c);
        }
        constexpr int kSeg = G::kTileN / 32;
        uint32_t r[2][16 * kSeg];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if constexpr (kSeg == 4)
            tc_ld_16x256b_x16(lane_base + (uint32_t(16 * h) << 16), r[h]);
          else
            tc_ld_16x256b_x4(lane_base + (uint32_t(16 * h) << 16), r[h]);
        }
        tc_wait_ld();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            store_row<OUT, kSeg>(r[h], e, pp, row0 + 16 * h + 8 * e, nt * G::kTileN, lane & 3,
                                 cofs, dofs);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty_addr + uint32_t(abuf * sizeof(uint64_t)));
      }
    }
    // this warp's TMA stores of D have completed before the CTA (and its shared memory) ends
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (kPair) cluster_sync();
  tc_fence_after();
  if (warp == 1) {
    if constexpr (kPair)
      tmem_dealloc_pair(tmem, kTmemCols);
    else
      tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort && p.status != nullptr) atomicOr(p.status, kDevTimeout);
}

// One problem (or a strided batch of equal problems).
template <int ESZ, int OUT, bool kPair, bool kNarrow, bool kHalfN>
__global__ void __launch_bounds__(Geo<ESZ, kPair, kNarrow, kHalfN>::kThreads, 1)
    spmma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                 const __grid_constant__ MmaParams p, const uint32_t idesc, const int staged) {
  // staged: the CTA-pair float epilogue moves C and D through shared memory by TMA
  spmma_body<ESZ, OUT, kPair, kNarrow, kHalfN, false>(&tmA, &tmB, &tmC, staged ? &tmD : nullptr, p,
                                                      idesc, nullptr);
}

// The problems of a group table, one persistent grid over all their tiles.
template <int ESZ, int OUT, bool kPair, bool kNarrow, bool kHalfN>
__global__ void __launch_bounds__(Geo<ESZ, kPair, kNarrow, kHalfN>::kThreads, 1)
    spmma_grouped_kernel(const __grid_constant__ MmaParams p,
                         const __grid_constant__ GroupTable gt) {
  spmma_body<ESZ, OUT, kPair, kNarrow, kHalfN, true>(nullptr, nullptr, nullptr, nullptr, p, 0u,
                                                     &gt);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D tensor map over `batch` row-major matrices: inner extent `cols` elements of `esz`
// bytes, `rows` rows, row pitch `pitch_bytes`, matrix pitch `batch_bytes`; box =
// box_cols x box_rows x 1.
bool make_tmap(CUtensorMap* m, const void* base, int esz, uint64_t cols, uint64_t rows,
               uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swz, uint64_t batch, uint64_t batch_bytes) {
  auto enc = get_encode();
  if (!enc) return false;
  const CUtensorMapDataType dt = esz == 4   ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                 : esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                            : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[3] = {cols, rows, batch};
  cuuint64_t strides[2] = {pitch_bytes, batch > 1 ? batch_bytes : rows * pitch_bytes};
  cuuint32_t box[3] = {box_cols, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The pair variant re-divides its registers with setmaxnreg, whose increase waits until
// the warpgroups' shares fit in what the block was launched with: refuse to launch a build
// whose register count would leave that wait unsatisfiable.
template <typename G, typename Kern>
bool register_split_fits(Kern kern) {
  cudaFuncAttributes fa;
  return cudaFuncGetAttributes(&fa, kern) == cudaSuccess &&
         uint64_t(fa.numRegs) * G::kThreads >= uint64_t(G::kRegsLight + G::kRegsEpi) * 256;
}

// Per-problem strides of the operands of a batched call (bytes).
struct BatchStrides {
  int64_t values, meta, b;
};

// The same instruction descriptor with half the MMA N (bits 17-22 hold N / 8).
inline uint32_t idesc_half_n(uint32_t id) {
  const uint32_t n = ((id >> 17) & 0x3Fu) << 3;
  return (id & ~(0x3Fu << 17)) | ((((n / 2) >> 3) & 0x3Fu) << 17);
}

template <int ESZ, int OUT, bool kPair, bool kNarrow = false, bool kHalfN = false>
int run(MmaParams p, const void* values, int64_t ldv, const void* meta, const void* B,
        int64_t ldb, uint32_t idesc, int num_sms, cudaStream_t s, const BatchStrides& bs) {
  using G = Geo<ESZ, kPair, kNarrow, kHalfN>;
  p.mtiles = (p.M + G::kTileM - 1) / G::kTileM;
  p.ntiles = (p.N + G::kTileN - 1) / G::kTileN;
  p.num_kb = (p.K + G::kStageK - 1) / G::kStageK;  // stages of this variant
  CUtensorMap tA, tB;
  memset(&tA, 0, sizeof(tA));
  memset(&tB, 0, sizeof(tB));
  p.meta = static_cast<const uint8_t*>(meta);
  p.stride_meta = bs.meta;
  if (p.K > 0) {  // with K == 0 no stage is loaded and the maps are never read
    const uint64_t nb = uint64_t(p.batch);
    if (!make_tmap(&tA, values, ESZ, uint64_t(p.K / 2), uint64_t(p.M), uint64_t(ldv) * ESZ,
                   128 / ESZ, 128, CU_TENSOR_MAP_SWIZZLE_128B, nb, uint64_t(bs.values)))
      return 4;
    if (!make_tmap(&tB, B, ESZ, uint64_t(p.N), uint64_t(p.K), uint64_t(ldb) * ESZ, G::kAtomN,
                   G::kStageK, kNarrow ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                   nb, uint64_t(bs.b)))
      return 4;
  }
  // the narrow variant loads only the B atoms that hold columns below N
  p.batoms = kNarrow ? (p.N + G::kAtomN - 1) / G::kAtomN : G::kAtoms;
  // CTA-pair products: C and D by TMA through the epilogue's staging boxes, 32 x 32
  // elements (f32 / s32 rows of 128 bytes with 128-byte swizzle, 16-bit rows of 64 bytes
  // with 64-byte swizzle)
  CUtensorMap tC, tD;
  memset(&tC, 0, sizeof(tC));
  memset(&tD, 0, sizeof(tD));
  int staged = 0;
  if constexpr (kPair) {
    const uint64_t nb = uint64_t(p.batch);
    const int dsz = OUT == 1 ? 2 : 4;  // f32 or s32 D: 4 bytes
    staged = make_tmap(&tD, p.D, dsz, uint64_t(p.N), uint64_t(p.M), uint64_t(p.ldd) * dsz, 32, 32,
                       dsz == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, nb,
                       uint64_t(p.stride_d) * dsz)
                 ? 1
                 : 0;
    if (staged && p.C != nullptr) {
      const int csz = p.ctype == 0 ? 4 : 2;
      staged = make_tmap(&tC, p.C, csz, uint64_t(p.N), uint64_t(p.M), uint64_t(p.ldc) * csz, 32,
                         32, csz == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B, nb,
                         uint64_t(p.stride_c) * csz)
                   ? 1
                   : 0;
    }
    if (!staged) return 4;
  }
  auto kern = spmma_kernel<ESZ, OUT, kPair, kNarrow, kHalfN>;
  if constexpr (kPair)
    if (!register_split_fits<G>(kern)) return 4;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes) !=
      cudaSuccess)
    return 4;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // may start during the previous kernel's tail; the kernel waits before touching data
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(G::kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const int tiles = p.mtiles * p.ntiles * p.batch;
  p.units = tiles;
  p.n_full = tiles;
  int units = num_sms;
  if (kPair) {
    cfg.gridDim = dim3(2 * (num_sms / 2), 1, 1);
    int max_clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, kern, &cfg) != cudaSuccess ||
        max_clusters < 1) {
      cudaGetLastError();
      max_clusters = num_sms / 2;
    }
    units = max_clusters;
  }
  if (tiles < units) units = tiles;
  // 16-bit float products on 256 x 256 pair tiles: when the last round of tiles would
  // leave more than half of the CTA pairs idle, its tiles run as two halves each (N / 2:
  // one B atom per CTA, half the MMA N), so the round takes about half as long
  if constexpr (kPair && !kHalfN && ESZ == 2 && OUT != 2) {
    const int rem = tiles % units;
    if (tiles > units && rem > 0 && 2 * rem <= units) {
      p.n_full = tiles - rem;
      p.units = p.n_full + 2 * rem;
      p.idesc_half = idesc_half_n(idesc);
    }
  }
  cfg.gridDim = dim3(units * (kPair ? 2 : 1), 1, 1);
  if (cudaLaunchKernelEx(&cfg, kern, tA, tB, tC, tD, p, idesc, staged) != cudaSuccess) return 4;
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

template <int ESZ, int OUT>
int dispatch(const MmaParams& p, const void* values, int64_t ldv, const void* meta,
             const void* B, int64_t ldb, uint32_t at, uint32_t bt, int num_sms, cudaStream_t s,
             const BatchStrides& bs) {
  if (p.N > 128)  // wide outputs: 256 x 256 tiles on CTA pairs
    return run<ESZ, OUT, true>(p, values, ldv, meta, B, ldb, idesc_sparse_f32(at, bt, 256, 256),
                               num_sms, s, bs);
  if (p.N <= 32) {  // skinny outputs: 128 x 32 tiles, MMA N = N rounded up to 16
    const uint32_t n_mma = uint32_t((p.N + 15) / 16 * 16);
    return run<ESZ, OUT, false, true>(p, values, ldv, meta, B, ldb,
                                      idesc_sparse_f32(at, bt, 128, n_mma), num_sms, s, bs);
  }
  // 16-bit operands, 32 < N <= 128: 256 x 128 tiles on CTA pairs (each CTA stages half of
  // B's columns, so a CTA moves 40 KB per stage instead of 56 KB; measured 4-8% faster than
  // 128 x 128 tiles on one CTA).  FP8: a half-width B (64 columns) is less than one
  // 128-byte swizzle atom, so 128 x 128 tiles on one CTA.
  if constexpr (ESZ == 2)
    return run<ESZ, OUT, true, false, true>(p, values, ldv, meta, B, ldb,
                                            idesc_sparse_f32(at, bt, 256, 128), num_sms, s, bs);
  else
    return run<ESZ, OUT, false>(p, values, ldv, meta, B, ldb,
                                idesc_sparse_f32(at, bt, 128, 128), num_sms, s, bs);
}

}  // namespace

int64_t int_ws_ldb(int64_t N) { return (N + 7) / 8 * 8; }

size_t int_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  const int64_t a = (M * (K / 2) * 2 + 255) / 256 * 256;
  const int64_t b = K * int_ws_ldb(N) * 2;
  return size_t(a + b);
}

namespace {

// One launch over up to kMaxGroup problems (already validated, all non-empty): a group
// table with each problem's tensor maps, tile range and epilogue fields.
template <int ESZ, int OUT, bool kPair, bool kNarrow = false, bool kHalfN = false>
int run_grouped(MmaParams p, const sp24_mma_problem* pr, int count, uint32_t at, uint32_t bt,
                int stage_k, int num_sms, cudaStream_t s) {
  using G = Geo<ESZ, kPair, kNarrow, kHalfN>;
  GroupTable gt;
  memset(&gt, 0, sizeof(gt));
  gt.count = count;
  int tiles = 0;
  for (int g = 0; g < count; ++g) {
    const sp24_mma_problem& q = pr[g];
    const int M = int(q.M), N = int(q.N), K = int(q.K);
    gt.M[g] = M;
    gt.N[g] = N;
    gt.K[g] = K;
    gt.num_kb[g] = (K + G::kStageK - 1) / G::kStageK;
    gt.img_kb[g] = (K + stage_k - 1) / stage_k;
    gt.mtiles[g] = (M + G::kTileM - 1) / G::kTileM;
    gt.ntiles[g] = (N + G::kTileN - 1) / G::kTileN;
    gt.batoms[g] = kNarrow ? (N + G::kAtomN - 1) / G::kAtomN : G::kAtoms;
    gt.idesc[g] = kNarrow ? idesc_sparse_f32(at, bt, 128, uint32_t((N + 15) / 16 * 16))
                          : idesc_sparse_f32(at, bt, kPair ? 256 : 128, uint32_t(G::kTileN));
    gt.C[g] = q.C;
    gt.D[g] = q.D;
    gt.meta[g] = static_cast<const uint8_t*>(q.meta);
    gt.ldc[g] = q.ldc;
    gt.ldd[g] = q.ldd;
    gt.c32[g] = (reinterpret_cast<uintptr_t>(q.C) % 32 == 0 && (q.ldc * 4) % 32 == 0) ? 1 : 0;
    gt.d32[g] = (reinterpret_cast<uintptr_t>(q.D) % 32 == 0 && (q.ldd * 4) % 32 == 0) ? 1 : 0;
    if (K > 0) {
      if (!make_tmap(&gt.a[g], q.values, ESZ, uint64_t(K / 2), uint64_t(M),
                     uint64_t(q.ldv) * ESZ, 128 / ESZ, 128, CU_TENSOR_MAP_SWIZZLE_128B, 1, 0) ||
          !make_tmap(&gt.b[g], q.B, ESZ, uint64_t(N), uint64_t(K), uint64_t(q.ldb) * ESZ,
                     G::kAtomN, G::kStageK,
                     kNarrow ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B, 1, 0))
        return 4;
    }
    gt.tile_start[g] = tiles;
    tiles += gt.mtiles[g] * gt.ntiles[g];
  }
  gt.tile_start[count] = tiles;
  auto kern = spmma_grouped_kernel<ESZ, OUT, kPair, kNarrow, kHalfN>;
  if constexpr (kPair)
    if (!register_split_fits<G>(kern)) return 4;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes) !=
      cudaSuccess)
    return 4;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kPair ? 2 : 1;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(G::kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::kSmemBytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  int units = kPair ? num_sms / 2 : num_sms;
  if (tiles < units) units = tiles;
  cfg.gridDim = dim3(units * (kPair ? 2 : 1), 1, 1);
  if (cudaLaunchKernelEx(&cfg, kern, p, gt) != cudaSuccess) return 4;
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

// The tile shape is the one sp24_mma picks for the widest output of the group, so that
// every problem fits it.
template <int ESZ, int OUT>
int dispatch_grouped(const MmaParams& p, const sp24_mma_problem* pr, int count, uint32_t at,
                     uint32_t bt, int stage_k, int num_sms, cudaStream_t s) {
  int64_t nmax = 0;
  for (int g = 0; g < count; ++g) nmax = pr[g].N > nmax ? pr[g].N : nmax;
  if (nmax > 128) return run_grouped<ESZ, OUT, true>(p, pr, count, at, bt, stage_k, num_sms, s);
  if (nmax <= 32)
    return run_grouped<ESZ, OUT, false, true>(p, pr, count, at, bt, stage_k, num_sms, s);
  if constexpr (ESZ == 2)
    return run_grouped<ESZ, OUT, true, false, true>(p, pr, count, at, bt, stage_k, num_sms, s);
  else
    return run_grouped<ESZ, OUT, false>(p, pr, count, at, bt, stage_k, num_sms, s);
}

}  // namespace

int launch_spmma_grouped(int ta, int tb, int tc, int td, const sp24_mma_problem* problems,
                         int count, int32_t* status, int num_sms, cudaStream_t s) {
  if (count <= 0) return 0;
  MmaParams p;
  memset(&p, 0, sizeof(p));
  p.batch = 1;
  p.status = status;
  p.chunk = 8;
  p.limit_ns = 1000000000ull;
  bool anyC = false;
  int64_t nmax = 0;
  for (int g = 0; g < count; ++g) {
    anyC = anyC || problems[g].C != nullptr;
    nmax = problems[g].N > nmax ? problems[g].N : nmax;
  }
  p.band_rows = band_rows_for(nmax);
  p.ctype = (anyC && tc == kBF16) ? 1 : (anyC && tc == kF16) ? 2 : 0;
  p.d_f16 = td == kF16 ? 1 : 0;
  const uint32_t at = (ta == kBF16 || ta == kE5M2) ? 1u : 0u;
  const uint32_t bt = (tb == kBF16 || tb == kE5M2) ? 1u : 0u;
  const bool out16 = td != kF32;
  const int sk = stage_k(ta);
  if (dtype_bytes(ta) == 2)
    return out16 ? dispatch_grouped<2, 1>(p, problems, count, at, bt, sk, num_sms, s)
                 : dispatch_grouped<2, 0>(p, problems, count, at, bt, sk, num_sms, s);
  return out16 ? dispatch_grouped<1, 1>(p, problems, count, at, bt, sk, num_sms, s)
               : dispatch_grouped<1, 0>(p, problems, count, at, bt, sk, num_sms, s);
}

int launch_spmma(int ta, int tb, int tc, int td, int64_t M, int64_t N, int64_t K,
                 const void* values, int64_t ldv, const void* meta, const void* B, int64_t ldb,
                 const void* C, int64_t ldc, void* D, int64_t ldd, void* workspace,
                 int32_t* status, int num_sms, cudaStream_t s, const BatchArgs* batch,
                 const uint32_t* index, int64_t ldi, uint64_t diag_stall_ns) {
  MmaParams p;
  memset(&p, 0, sizeof(p));
  p.index = index;  // canonical index instead of the image (one problem only)
  p.ldi = ldi;
  p.idx_vec = (index != nullptr && reinterpret_cast<uintptr_t>(index) % 16 == 0 && ldi % 4 == 0) ? 1 : 0;
  BatchStrides bs{0, 0, 0};
  p.batch = 1;
  if (batch != nullptr && batch->count > 1) {
    p.batch = int(batch->count);
    bs.values = ld_bytes(ta, batch->stride_values);
    bs.meta = batch->stride_meta;
    bs.b = ld_bytes(tb, batch->stride_b);
    p.stride_c = batch->stride_c;
    p.stride_d = batch->stride_d;
  }
  p.C = C;
  p.D = D;
  p.ldc = ldc;
  p.ldd = ldd;
  p.status = status;
  // 32-byte vector accesses need a 32-byte aligned base and pitch (the ABI promises 16)
  p.c32 = (reinterpret_cast<uintptr_t>(C) % 32 == 0 && (ldc * 4) % 32 == 0) ? 1 : 0;
  p.ctype = (C != nullptr && tc == kBF16) ? 1 : (C != nullptr && tc == kF16) ? 2 : 0;
  p.d_f16 = td == kF16 ? 1 : 0;
  p.d32 = (reinterpret_cast<uintptr_t>(D) % 32 == 0 && (ldd * 4) % 32 == 0) ? 1 : 0;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.mtiles = p.ntiles = 0;
  p.img_kb = int((K + stage_k(ta) - 1) / stage_k(ta));  // metadata image stages per tile
  p.num_kb = p.img_kb;  // the variant's own stage count is set at launch
  p.limit_ns = 1000000000ull;  // 1 s per wait
  p.band_rows = band_rows_for(N);
  if (diag_stall_ns != 0) {  // give-up self-test: no copies, short waits
    p.diag_stall = 1;
    p.limit_ns = diag_stall_ns;
  }
  if (is_int(ta)) {
    // integers: widen both operands to bf16 (exact) and run the bf16 tensor path with
    // chunked integer accumulation on 256 x 256 tiles (the MMA waits for each chunk's
    // drain, which is short against a chunk of 8 to 64 stages)
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    uint8_t* wa = ws;
    uint8_t* wb = ws + (M * (K / 2) * 2 + 255) / 256 * 256;
    const int64_t ldbw = int_ws_ldb(N);
    if (K > 0) {
      if (launch_widen(values, ld_bytes(ta, ldv), wa, K / 2, M, K / 2, is_signed_int(ta),
                       elem_bits(ta), num_sms, s) != cudaSuccess ||
          launch_widen(B, ld_bytes(tb, ldb), wb, ldbw, K, N, is_signed_int(tb), elem_bits(tb),
                       num_sms, s) != cudaSuccess)
        return 4;
    }
    p.chunk = (ta == kS8 && tb == kS8) ? 16 : is_i4(ta) ? 64 : 8;
    // kind::f16 with bf16 operands: type code 1 for A and B
    return run<2, 2, true>(p, wa, K / 2, meta, wb, ldbw, idesc_sparse_f32(1, 1, 256, 256),
                           num_sms, s, bs);
  }
  const int esz = dtype_bytes(ta);
  // kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = E4M3, 1 = E5M2
  const uint32_t at = (ta == kBF16 || ta == kE5M2) ? 1u : 0u;
  const uint32_t bt = (tb == kBF16 || tb == kE5M2) ? 1u : 0u;
  const bool out16 = td != kF32;  // bf16 or f16 (p.d_f16)
  if (esz == 2)
    return out16 ? dispatch<2, 1>(p, values, ldv, meta, B, ldb, at, bt, num_sms, s, bs)
                    : dispatch<2, 0>(p, values, ldv, meta, B, ldb, at, bt, num_sms, s, bs);
  return out16 ? dispatch<1, 1>(p, values, ldv, meta, B, ldb, at, bt, num_sms, s, bs)
                  : dispatch<1, 0>(p, values, ldv, meta, B, ldb, at, bt, num_sms, s, bs);
}

}  // namespace sp24
