// spmma.cu -- the 2:4 sparse GEMM D = expand(A_c, meta) * B + C on sm_103a tensor cores.
//
// Semantics: "RDNA4 sparse WMMA builtins", "Builtin reference" (each builtin returns
// expand(srcA, index) x srcB + srcC, f32 accumulate); "v_smfmac_f32_32x32x32_bf8_bf8",
// "Semantics" (D = A(sparse) * B + D).  The pages' kernels issue one 16x16 (or 32x32)
// builtin per wavefront per K step from LDS tiles; here one elected thread per CTA issues
// tcgen05.mma.sp on a 128 x BN tile held in tensor memory.
//
// Structure (one CTA per SM, persistent over output tiles, 6 warps):
//   warp 0     TMA producer: per K stage, one 128x128-byte box of compressed A
//              (K-major, 128-byte swizzle), BN/atom boxes of B (K x N row-major =
//              MN-major, 128-byte swizzle) and one contiguous block of the metadata
//              image (cp.async.bulk), all completing on the stage's "full" mbarrier.
//   warp 1     TMEM owner + MMA issuer: copies the stage's metadata smem -> TMEM
//              (tcgen05.cp), issues 4 tcgen05.mma.sp, and tcgen05.commit releases the
//              stage; after the last stage it commits the accumulator buffer.
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes, + C, cast, store; then free
//              the accumulator buffer.  Accumulators are double-buffered in TMEM, so
//              the epilogue of tile t overlaps the main loop of tile t+1.
// Every mbarrier wait is bounded (see mbar_wait); a wait that gives up sets
// SP24_DEV_TIMEOUT in the caller's status word and the CTA drains and exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "sp24_device.cuh"
#include "sp24_internal.h"

namespace sp24 {
namespace {

constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kABytes = 128 * 128;  // one stage of compressed A: 128 rows x 128 bytes

struct MmaParams {
  const uint8_t* meta;
  const void* C;
  void* D;
  int64_t ldc, ldd;
  int32_t* status;
  int M, N, K;
  int mtiles, ntiles, num_kb;
  uint64_t limit_ns;
};

template <int ESZ, int BN>
struct Geo {
  static constexpr int kStageK = ESZ == 2 ? 128 : 256;          // dense K per stage
  static constexpr int kMmaK = ESZ == 2 ? 32 : 64;               // dense K per MMA
  static constexpr int kMmas = kStageK / kMmaK;                  // 4
  static constexpr int kMetaBytes = kMmas * kMetaBlockBytes;     // 4 blocks of 2 KB
  static constexpr int kMetaSlotCols = 16;                       // TMEM columns per MMA slot
  static constexpr int kAtomN = 128 / ESZ;                       // N elements per 128 B
  static constexpr int kAtoms = BN / kAtomN;
  static constexpr int kAtomBytes = kStageK * 128;               // one B box
  static constexpr int kBBytes = kAtoms * kAtomBytes;
  static constexpr int kStageBytes = kABytes + kBBytes + kMetaBytes;
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static constexpr uint32_t kTx = kABytes + kBBytes + kMetaBytes;
  static constexpr uint32_t kMetaTmemCol = 2 * BN;               // after both accumulators
  static_assert(BN % kAtomN == 0, "BN must be a multiple of the swizzle atom");
  static_assert(2 * BN + kStages * kMmas * kMetaSlotCols <= int(kTmemCols), "TMEM budget");
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

// OUT: 0 = f32, 1 = bf16, 2 = s32 (reserved).  C (if present) is f32 for float paths.
template <int ESZ, int BN, int OUT>
__global__ void __launch_bounds__(kThreads, 1)
    spmma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                 const MmaParams p, const uint32_t idesc) {
  using G = Geo<ESZ, BN>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  __shared__ __align__(8) uint64_t full_bar[kStages], empty_bar[kStages];
  __shared__ __align__(8) uint64_t acc_full[2], acc_empty[2], drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint8_t* sM = sB + kStages * G::kBBytes;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const int ntiles_total = p.mtiles * p.ntiles;
  volatile int* abort = &abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < ntiles_total && !*abort; t += gridDim.x) {
        const int mt = t % p.mtiles, nt = t / p.mtiles;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort, p.limit_ns)) break;
          mbar_arrive_expect_tx(&full_bar[stage], G::kTx);
          tma_load_2d(sA + stage * kABytes, &tmA, &full_bar[stage], kb * (G::kStageK / 2),
                      mt * 128);
#pragma unroll
          for (int a = 0; a < G::kAtoms; ++a)
            tma_load_2d(sB + stage * G::kBBytes + a * G::kAtomBytes, &tmB, &full_bar[stage],
                        nt * BN + a * G::kAtomN, kb * G::kStageK);
          bulk_load(sM + stage * G::kMetaBytes,
                    p.meta + (int64_t(mt) * p.num_kb + kb) * G::kMetaBytes, G::kMetaBytes,
                    &full_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (*abort) {
        // give copies already issued time to land before the CTA can exit
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t adesc_hi = smem_desc_hi(16, 1024, 2);
      const uint64_t bdesc_hi = smem_desc_hi(G::kAtomBytes, 1024, 2);
      const uint64_t mdesc_hi = smem_desc_hi(0, 128, 0);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      for (int t = blockIdx.x; t < ntiles_total && !*abort; t += gridDim.x, ++local) {
        const int abuf = local & 1;
        const uint32_t acc_parity = ((local >> 1) & 1) ^ 1u;
        if (!mbar_wait(&acc_empty[abuf], acc_parity, abort, p.limit_ns)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + uint32_t(abuf * BN);
        bool ok = true;
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort, p.limit_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // metadata: MMA j of this stage reads the 16-column-aligned slot (stage, j)
          const uint32_t e_tmem =
              tmem + G::kMetaTmemCol + uint32_t(stage * G::kMmas * G::kMetaSlotCols);
          const uint32_t m_saddr = smem_addr(sM + stage * G::kMetaBytes);
#pragma unroll
          for (int j = 0; j < G::kMmas; ++j)
            tc_cp_128x128b(e_tmem + j * G::kMetaSlotCols,
                           smem_desc(m_saddr + j * kMetaBlockBytes, mdesc_hi));
          const uint32_t a_saddr = smem_addr(sA + stage * kABytes);
          const uint32_t b_saddr = smem_addr(sB + stage * G::kBBytes);
          const int k0 = kb * G::kStageK;
#pragma unroll
          for (int j = 0; j < G::kMmas; ++j) {
            if (k0 + j * G::kMmaK < p.K) {
              tc_mma_sp<ESZ == 1>(d_tmem, smem_desc(a_saddr + 32 * j, adesc_hi),
                                  smem_desc(b_saddr + j * G::kMmaK * 128, bdesc_hi),
                                  e_tmem + j * G::kMetaSlotCols, idesc,
                                  (kb > 0 || j > 0) ? 1u : 0u);
            }
          }
          tc_commit(&empty_bar[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&acc_full[abuf]);
      }
      // all MMAs issued by this thread complete before TMEM can be released
      tc_commit(&drain_bar);
      mbar_wait_drain(&drain_bar, 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    int local = 0;
    for (int t = blockIdx.x; t < ntiles_total; t += gridDim.x, ++local) {
      const int mt = t % p.mtiles, nt = t / p.mtiles;
      const int abuf = local & 1;
      if (!mbar_wait(&acc_full[abuf], (local >> 1) & 1, abort, p.limit_ns)) break;
      tc_fence_after();
      const int row = mt * 128 + quad * 32 + lane;
      const bool row_ok = row < p.M;
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tc_ld_32x32b_x32(tmem + (uint32_t(quad * 32) << 16) + uint32_t(abuf * BN + c * 32), r);
        tc_wait_ld();
        const int col0 = nt * BN + c * 32;
        if (!row_ok || col0 >= p.N) continue;
        float v[32];
        if (p.K > 0) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = 0.f;
        }
        const bool full = col0 + 32 <= p.N;
        if (p.C != nullptr) {
          const float* crow = static_cast<const float*>(p.C) + int64_t(row) * p.ldc + col0;
          if (full) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              const float4 cv = __ldcs(reinterpret_cast<const float4*>(crow + j));
              v[j] += cv.x;
              v[j + 1] += cv.y;
              v[j + 2] += cv.z;
              v[j + 3] += cv.w;
            }
          } else {
            for (int j = 0; j < 32 && col0 + j < p.N; ++j) v[j] += crow[j];
          }
        }
        if constexpr (OUT == 0) {
          float* drow = static_cast<float*>(p.D) + int64_t(row) * p.ldd + col0;
          if (full) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              __stcs(reinterpret_cast<float4*>(drow + j), make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]));
          } else {
            for (int j = 0; j < 32 && col0 + j < p.N; ++j) drow[j] = v[j];
          }
        } else {
          __nv_bfloat16* drow = static_cast<__nv_bfloat16*>(p.D) + int64_t(row) * p.ldd + col0;
          if (full) {
#pragma unroll
            for (int j = 0; j < 32; j += 8) {
              __nv_bfloat162 h0 = __floats2bfloat162_rn(v[j], v[j + 1]);
              __nv_bfloat162 h1 = __floats2bfloat162_rn(v[j + 2], v[j + 3]);
              __nv_bfloat162 h2 = __floats2bfloat162_rn(v[j + 4], v[j + 5]);
              __nv_bfloat162 h3 = __floats2bfloat162_rn(v[j + 6], v[j + 7]);
              uint4 u;
              memcpy(&u.x, &h0, 4);
              memcpy(&u.y, &h1, 4);
              memcpy(&u.z, &h2, 4);
              memcpy(&u.w, &h3, 4);
              __stcs(reinterpret_cast<uint4*>(drow + j), u);
            }
          } else {
            for (int j = 0; j < 32 && col0 + j < p.N; ++j) drow[j] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[abuf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && *abort && p.status != nullptr) atomicOr(p.status, kDevTimeout);
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

// 2-D tensor map over a row-major matrix: inner extent `cols` elements of `esz` bytes,
// `rows` rows, row pitch `pitch_bytes`; box = box_cols x box_rows, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, int esz, uint64_t cols, uint64_t rows,
               uint64_t pitch_bytes, uint32_t box_cols, uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      esz == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int ESZ, int BN, int OUT>
int run(const MmaParams& p, const void* values, int64_t ldv, const void* B, int64_t ldb,
        uint32_t idesc, int num_sms, cudaStream_t s) {
  using G = Geo<ESZ, BN>;
  CUtensorMap tA, tB;
  memset(&tA, 0, sizeof(tA));
  memset(&tB, 0, sizeof(tB));
  if (p.K > 0) {  // with K == 0 no stage is loaded and the maps are never read
    if (!make_tmap(&tA, values, ESZ, uint64_t(p.K / 2), uint64_t(p.M), uint64_t(ldv) * ESZ,
                   128 / ESZ, 128))
      return 4;
    if (!make_tmap(&tB, B, ESZ, uint64_t(p.N), uint64_t(p.K), uint64_t(ldb) * ESZ, G::kAtomN,
                   G::kStageK))
      return 4;
  }
  auto kern = spmma_kernel<ESZ, BN, OUT>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmemBytes) !=
      cudaSuccess)
    return 4;
  const int tiles = p.mtiles * p.ntiles;
  const int grid = tiles < num_sms ? tiles : num_sms;
  kern<<<grid, kThreads, G::kSmemBytes, s>>>(tA, tB, p, idesc);
  return cudaGetLastError() == cudaSuccess ? 0 : 4;
}

}  // namespace

int launch_spmma(int ta, int tb, int tc, int td, int64_t M, int64_t N, int64_t K,
                 const void* values, int64_t ldv, const void* meta, const void* B, int64_t ldb,
                 const void* C, int64_t ldc, void* D, int64_t ldd, int32_t* status,
                 int num_sms, cudaStream_t s) {
  (void)tc;
  const int esz = dtype_bytes(ta);
  MmaParams p;
  p.meta = static_cast<const uint8_t*>(meta);
  p.C = C;
  p.D = D;
  p.ldc = ldc;
  p.ldd = ldd;
  p.status = status;
  p.M = int(M);
  p.N = int(N);
  p.K = int(K);
  p.mtiles = int((M + 127) / 128);
  const int stage_k = esz == 2 ? 128 : 256;
  p.num_kb = int((K + stage_k - 1) / stage_k);
  p.limit_ns = 1000000000ull;  // 1 s per wait
  constexpr int BN = 128;
  p.ntiles = int((N + BN - 1) / BN);
  // kind::f16: 0 = f16, 1 = bf16; kind::f8f6f4: 0 = E4M3, 1 = E5M2
  const uint32_t at = (ta == kBF16 || ta == kE5M2) ? 1u : 0u;
  const uint32_t bt = (tb == kBF16 || tb == kE5M2) ? 1u : 0u;
  const uint32_t idesc = idesc_sparse_f32(at, bt, 128, BN);
  const bool out_bf16 = td == kBF16;
  if (esz == 2)
    return out_bf16 ? run<2, BN, 1>(p, values, ldv, B, ldb, idesc, num_sms, s)
                    : run<2, BN, 0>(p, values, ldv, B, ldb, idesc, num_sms, s);
  return out_bf16 ? run<1, BN, 1>(p, values, ldv, B, ldb, idesc, num_sms, s)
                  : run<1, BN, 0>(p, values, ldv, B, ldb, idesc, num_sms, s);
}

}  // namespace sp24
