// noalloc.cu -- sp24_mma_i8_noalloc: the 8-bit integer sparse product with its scratch in
// a fixed device array instead of a caller-provided workspace.
//
// Some callers cannot allocate device memory when they call the product: a plugin that
// runs inside a host framework owning all device memory and handing out no workspace, or
// a caller with a fixed memory plan that forbids allocations after start-up (cudaMalloc
// may also synchronise the device, which a latency-bound caller cannot afford).  This
// entry point needs nothing from them but inputs and outputs.
//
// The scratch is one file-scope device array of SP24_NOALLOC_SCRATCH_BYTES; every GPU that
// loads the library holds it until the process exits.  All calls share it: each call
// writes the part it uses (the two operands widened to bf16) before reading it, so nothing
// has to start at zero, and the array keeps the last call's contents.  Two calls whose
// work overlaps on the GPU (different streams, no ordering between them) race on it.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/sp24.h"
#include "sp24_internal.h"

namespace sp24 {
namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[SP24_NOALLOC_SCRATCH_BYTES];

// The current context's unique id (cuCtxGetId through the runtime's driver entry
// point, so the library needs no link against the driver library), or 0 if unavailable.
unsigned long long current_context_id() {
  using GetCurrent = CUresult (*)(CUcontext*);
  using GetId = CUresult (*)(CUcontext, unsigned long long*);
  static GetCurrent get_current = nullptr;
  static GetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrent>(f);
    f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetId>(f);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS ||
      ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the array in the current context of device `dev` (which must be
// current).  In host code the array's name is only a stand-in, never a device address.
// The address is looked up once per device and context: a context created anew (after
// cudaDeviceReset, for example) has a different id, and its first call looks it up again.
void* scratch_address(int dev) {
  static std::mutex mu;
  static void* addr[64];
  static unsigned long long ctx_of[64];
  if (dev < 0 || dev >= 64) return nullptr;
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx_of[dev] != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return nullptr;
    }
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace sp24

using namespace sp24;

extern "C" sp24_status sp24_mma_i8_noalloc(sp24_dtype ta, sp24_dtype tb, sp24_dtype tc,
                                           sp24_dtype td, int64_t M, int64_t N, int64_t K,
                                           const void* values, int64_t ldv, const void* meta,
                                           const void* B, int64_t ldb, const void* C,
                                           int64_t ldc, void* D, int64_t ldd,
                                           int32_t* d_status, void* stream) {
  if (!is_i8(ta) || tb != SP24_S8 || td != SP24_S32) return SP24_ERR_UNSUPPORTED;
  if (C != nullptr && tc != SP24_S32) return SP24_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 0 || (K % 32) != 0) return SP24_ERR_INVALID_ARG;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return SP24_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return SP24_OK;
  if (!D || (K > 0 && (!values || !meta || !B))) return SP24_ERR_INVALID_ARG;
  if (ldd < N || (C && ldc < N) || (K > 0 && (ldv < K / 2 || ldb < N)))
    return SP24_ERR_INVALID_ARG;
  if (int_workspace_bytes(M, N, K) > size_t(SP24_NOALLOC_SCRATCH_BYTES))
    return SP24_ERR_SCRATCH_TOO_SMALL;
  if (!aligned16(D) || (ldd * 4) % 16) return SP24_ERR_ALIGN;
  if (C && (!aligned16(C) || (ldc * 4) % 16)) return SP24_ERR_ALIGN;
  if (K > 0 && (!aligned16(values) || !aligned16(meta) || !aligned16(B) || ldv % 16 || ldb % 16))
    return SP24_ERR_ALIGN;
  int sms = 0;
  if (!current_device(&sms)) return SP24_ERR_NO_DEVICE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SP24_ERR_CUDA;
  }
  void* scratch = scratch_address(dev);
  if (scratch == nullptr) return SP24_ERR_CUDA;
  const int rc = launch_spmma(ta, tb, tc, td, M, N, K, values, ldv, meta, B, ldb, C, ldc, D, ldd,
                              scratch, d_status, sms, static_cast<cudaStream_t>(stream));
  return static_cast<sp24_status>(rc);
}
