// sp24_device.cuh -- inline-PTX building blocks for the sm_103a kernels of libsp24:
// mbarriers with bounded waits, TMA (cp.async.bulk[.tensor]) loads, and the tcgen05
// family (TMEM allocation, tcgen05.st, tcgen05.mma.sp, tcgen05.commit, tcgen05.ld).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace sp24 {

// Device status bits (same values as SP24_DEV_* in include/sp24.h).
constexpr int kDevNot24 = 1;
constexpr int kDevTimeout = 2;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n.reg .b64 st;\nmbarrier.arrive.shared::cta.b64 st, [%0];\n}\n" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n.reg .b64 st;\nmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n}\n" ::"r"(
          smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n.reg .pred P;\nmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n"
      "selp.b32 %0, 1, 0, P;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up after
// `limit_ns` of wall time or as soon as *abort becomes non-zero (another role gave up);
// on giving up it sets *abort and returns false.  Never spins forever.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag: used to let operations already in flight
// (bulk copies, MMAs) finish before their shared or tensor memory is released.
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 0u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Programmatic dependent launch: a kernel launched with programmatic stream serialization
// may start while the kernel before it on the stream is still running; griddep_wait()
// returns once that kernel has completed and its memory writes are visible.  A kernel that
// calls griddep_launch_dependents() lets the next such kernel start early (its blocks are
// placed as resources free up; it still waits before touching data).
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA / bulk copies
__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// TMA 3-D load (x, y and a batch coordinate z).
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const void* tmap, uint64_t* bar,
                                            int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_addr(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// TMA 3-D store of a shared-memory box to global memory (elements outside the tensor are
// not written), tracked by this thread's bulk async-group.
__device__ __forceinline__ void tma_store_3d(const void* tmap, const void* smem_src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(smem_addr(smem_src)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until this thread's committed bulk stores have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// wait until this thread's committed bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// order this thread's generic-proxy shared-memory writes before later async-proxy (TMA)
// reads of them
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Start pulling `bytes` (multiple of 16) of global memory at a 16-byte aligned address
// into L2; no completion is tracked and nothing is written to shared memory.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(gsrc)),
               "r"(bytes)
               : "memory");
}

// Fetch one box of a tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const void* tmap, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(smem_slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// One sparse MMA, cta_group::1: D[tmem] (+)= expand(A[smem], meta[tmem]) * B[smem].
template <bool kF8>
__device__ __forceinline__ void tc_mma_sp(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                          uint32_t e_tmem, uint32_t idesc, uint32_t accumulate) {
  if constexpr (kF8) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.sp.cta_group::1.kind::f8f6f4 [%0], %1, %2, [%3], %4, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(e_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.sp.cta_group::1.kind::f16 [%0], %1, %2, [%3], %4, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(e_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this thread is done.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// Store one 32-bit column (x1) or two consecutive columns (x2) of the warp's 32 lanes:
// thread t writes lane (base lane + t).
__device__ __forceinline__ void tc_st_32x32b_x1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void tc_st_32x32b_x2(uint32_t taddr, uint32_t v0, uint32_t v1) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x2.b32 [%0], {%1, %2};" ::"r"(taddr), "r"(v0),
               "r"(v1)
               : "memory");
}
__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Per-warpgroup register reallocation (all 128 threads of the warpgroup execute it).
template <uint32_t kRegs>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// 32 lanes x 32 consecutive 32-bit columns: thread t gets lane (base lane + t).
__device__ __forceinline__ void tc_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// 16 lanes x 8N columns (.16x256b.xN): for repetition i (columns 8i .. 8i+7) thread t
// gets lane (base + t/4), columns 8i + 2(t%4) and +1, in r[4i], r[4i+1], and lane
// (base + 8 + t/4), the same two columns, in r[4i+2], r[4i+3].
__device__ __forceinline__ void tc_ld_16x256b_x4(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_16x256b_x16(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
}
// 32 lanes x 16 consecutive 32-bit columns: thread t gets lane (base lane + t).
__device__ __forceinline__ void tc_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- CTA pairs (cluster of 2)
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
// Arrive on an mbarrier given by its shared::cluster address (possibly in the peer CTA),
// with the instruction's default semantics (release at CTA scope).  Every use follows
// completed tensor-memory work of this thread (tcgen05.wait::st or ::ld) and a
// tcgen05.fence::before_thread_sync, which orders that work before the arrive for the
// thread that waits on the barrier and then issues tcgen05 operations.  A release at
// cluster scope is not needed for that and was measured to stall: as the writers'
// per-stage arrive it made the CTA-pair GEMM 1.7x slower (bf16 4096^3: 157 us against
// 92 us).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA 3-D load into this CTA's shared memory whose completion is counted on an mbarrier
// of either CTA of the pair (.cta_group::2), given by its shared::cluster address.
__device__ __forceinline__ void tma_load_3d_pair(void* smem_dst, const void* tmap, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(smem_slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// Sparse MMA across the CTA pair (M = 256: 128 rows of A and half of B's N in each CTA).
template <bool kF8>
__device__ __forceinline__ void tc_mma_sp_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t e_tmem, uint32_t idesc,
                                               uint32_t accumulate) {
  if constexpr (kF8) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.sp.cta_group::2.kind::f8f6f4 [%0], %1, %2, [%3], %4, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(e_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %5, 0;\n"
        "tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(e_tmem), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}
// arrive (once the pair's prior tcgen05 work is done) on the barrier at the same offset
// in every CTA of `mask`
__device__ __forceinline__ void tc_commit_pair_mc(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// One whole stage of the main loop in a single instruction sequence: test (without
// waiting) whether the next stage's barrier phase `next_par` at shared address `next_bar`
// has completed, issue the stage's four sparse MMAs and the commit that arrives on the
// stage's empty barrier(s), and only then look at the test's outcome.  The issuing thread
// spends tens of cycles per tcgen05 instruction and over a hundred per barrier test, while
// four M = 256, N = 256 MMAs keep the tensor pipe busy for about 512 cycles; testing the
// next barrier while the MMAs are issued keeps its latency off the loop.
// MMA j reads A at descriptor a0 + j * a_step, B at b0 + j * b_step (descriptor units of 16
// bytes) and its metadata at TMEM column e0 + 16 j; acc0 = 0 starts the accumulation.
// kPair: cta_group::2 with a commit multicast to both CTAs of the pair (`mask`);
// otherwise cta_group::1 and a commit to the local barrier `empty_bar`.
// Returns whether the next stage's phase had completed at the test.
template <bool kPair, bool kF8>
__device__ __forceinline__ bool mma_stage_test_next(uint32_t next_bar, uint32_t next_par,
                                                    uint32_t d, uint64_t a0, uint64_t b0,
                                                    uint32_t a_step, uint32_t b_step,
                                                    uint32_t e0, uint32_t idesc, uint32_t acc0,
                                                    uint32_t empty_bar) {
  uint32_t ok;
#define SP24_STAGE_ASM(GROUP, KIND, COMMIT)                                                   \
  asm volatile(                                                                              \
      "{\n"                                                                                  \
      ".reg .pred pn, pa, pt;\n"                                                             \
      ".reg .b64 a1, a2, a3, b1, b2, b3, sa, sb;\n"                                          \
      ".reg .b32 e1, e2, e3;\n"                                                              \
      "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n"                            \
      "setp.ne.b32 pa, %10, 0;\n"                                                            \
      "setp.eq.b32 pt, %2, %2;\n"                                                            \
      "cvt.u64.u32 sa, %6;\n"                                                                \
      "cvt.u64.u32 sb, %7;\n"                                                                \
      "add.s64 a1, %4, sa;\n add.s64 a2, a1, sa;\n add.s64 a3, a2, sa;\n"                   \
      "add.s64 b1, %5, sb;\n add.s64 b2, b1, sb;\n add.s64 b3, b2, sb;\n"                   \
      "add.u32 e1, %8, 16;\n add.u32 e2, %8, 32;\n add.u32 e3, %8, 48;\n"                    \
      "tcgen05.mma.sp." GROUP "." KIND " [%3], %4, %5, [%8], %9, pa;\n"                      \
      "tcgen05.mma.sp." GROUP "." KIND " [%3], a1, b1, [e1], %9, pt;\n"                      \
      "tcgen05.mma.sp." GROUP "." KIND " [%3], a2, b2, [e2], %9, pt;\n"                      \
      "tcgen05.mma.sp." GROUP "." KIND " [%3], a3, b3, [e3], %9, pt;\n" COMMIT               \
      "selp.b32 %0, 1, 0, pn;\n"                                                             \
      "}\n"                                                                                  \
      : "=r"(ok)                                                                             \
      : "r"(next_bar), "r"(next_par), "r"(d), "l"(a0), "l"(b0), "r"(a_step), "r"(b_step),    \
        "r"(e0), "r"(idesc), "r"(acc0), "r"(empty_bar), "h"(uint16_t(3))                     \
      : "memory")
  if constexpr (kPair) {
    if constexpr (kF8)
      SP24_STAGE_ASM("cta_group::2", "kind::f8f6f4",
                     "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
                     "multicast::cluster.b64 [%11], %12;\n");
    else
      SP24_STAGE_ASM("cta_group::2", "kind::f16",
                     "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
                     "multicast::cluster.b64 [%11], %12;\n");
  } else {
    if constexpr (kF8)
      SP24_STAGE_ASM("cta_group::1", "kind::f8f6f4",
                     "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
                     "[%11];\n");
    else
      SP24_STAGE_ASM("cta_group::1", "kind::f16",
                     "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
                     "[%11];\n");
  }
#undef SP24_STAGE_ASM
  return ok != 0;
}

// The same for a stage of eight kind::f16 MMAs whose A spans two 128-byte swizzle boxes:
// MMAs 0-3 read A at a0 + j * a_step, MMAs 4-7 at a0 + a_box + (j - 4) * a_step; B at
// b0 + j * b_step; metadata at e0 + 16 j.  kPair: cta_group::2 with the commit multicast to
// both CTAs of the pair; otherwise cta_group::1 and a commit to the local barrier.
template <bool kPair>
__device__ __forceinline__ bool mma_stage8_test_next(uint32_t next_bar, uint32_t next_par,
                                                     uint32_t d, uint64_t a0, uint64_t b0,
                                                     uint32_t a_step, uint32_t a_box,
                                                     uint32_t b_step, uint32_t e0,
                                                     uint32_t idesc, uint32_t acc0,
                                                     uint32_t empty_bar) {
  uint32_t ok;
#define SP24_STAGE8_ASM(GROUP, COMMIT)                                                        \
  asm volatile(                                                                              \
      "{\n"                                                                                  \
      ".reg .pred pn, pa, pt;\n"                                                             \
      ".reg .b64 a1, a2, a3, a4, a5, a6, a7, b1, b2, b3, b4, b5, b6, b7, sa, sx, sb;\n"      \
      ".reg .b32 e1, e2, e3, e4, e5, e6, e7;\n"                                              \
      "mbarrier.test_wait.parity.shared::cta.b64 pn, [%1], %2;\n"                            \
      "setp.ne.b32 pa, %11, 0;\n"                                                            \
      "setp.eq.b32 pt, %2, %2;\n"                                                            \
      "cvt.u64.u32 sa, %6;\n"                                                                \
      "cvt.u64.u32 sx, %7;\n"                                                                \
      "cvt.u64.u32 sb, %8;\n"                                                                \
      "add.s64 a1, %4, sa;\n add.s64 a2, a1, sa;\n add.s64 a3, a2, sa;\n"                   \
      "add.s64 a4, %4, sx;\n add.s64 a5, a4, sa;\n add.s64 a6, a5, sa;\n"                   \
      "add.s64 a7, a6, sa;\n"                                                                \
      "add.s64 b1, %5, sb;\n add.s64 b2, b1, sb;\n add.s64 b3, b2, sb;\n"                   \
      "add.s64 b4, b3, sb;\n add.s64 b5, b4, sb;\n add.s64 b6, b5, sb;\n"                   \
      "add.s64 b7, b6, sb;\n"                                                                \
      "add.u32 e1, %9, 16;\n add.u32 e2, %9, 32;\n add.u32 e3, %9, 48;\n"                    \
      "add.u32 e4, %9, 64;\n add.u32 e5, %9, 80;\n add.u32 e6, %9, 96;\n"                    \
      "add.u32 e7, %9, 112;\n"                                                               \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], %4, %5, [%9], %10, pa;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a1, b1, [e1], %10, pt;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a2, b2, [e2], %10, pt;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a3, b3, [e3], %10, pt;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a4, b4, [e4], %10, pt;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a5, b5, [e5], %10, pt;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a6, b6, [e6], %10, pt;\n"                   \
      "tcgen05.mma.sp." GROUP ".kind::f16 [%3], a7, b7, [e7], %10, pt;\n" COMMIT            \
      "selp.b32 %0, 1, 0, pn;\n"                                                             \
      "}\n"                                                                                  \
      : "=r"(ok)                                                                             \
      : "r"(next_bar), "r"(next_par), "r"(d), "l"(a0), "l"(b0), "r"(a_step), "r"(a_box),     \
        "r"(b_step), "r"(e0), "r"(idesc), "r"(acc0), "r"(empty_bar), "h"(uint16_t(3))        \
      : "memory")
  if constexpr (kPair)
    SP24_STAGE8_ASM("cta_group::2",
                    "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster."
                    "multicast::cluster.b64 [%12], %13;\n");
  else
    SP24_STAGE8_ASM("cta_group::1",
                    "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
                    "[%12];\n");
#undef SP24_STAGE8_ASM
  return ok != 0;
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor: start address, leading / stride byte offsets,
// version 1 (bit 46), swizzle mode in bits 61-63 (0 none, 2 = 128-byte).
__host__ __device__ constexpr uint64_t smem_desc_hi(uint32_t lbo, uint32_t sbo, uint32_t swz) {
  return (uint64_t((lbo >> 4) & 0x3FFFu) << 16) | (uint64_t((sbo >> 4) & 0x3FFFu) << 32) |
         (uint64_t(1) << 46) | (uint64_t(swz & 7u) << 61);
}
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint64_t hi) {
  return hi | uint64_t((saddr >> 4) & 0x3FFFu);
}

// Instruction descriptor of a sparse MMA with f32 accumulate, A K-major, B MN-major.
// atype/btype: kind::f16 -> 0 f16, 1 bf16; kind::f8f6f4 -> 0 E4M3, 1 E5M2.
__host__ __device__ constexpr uint32_t idesc_sparse_f32(uint32_t atype, uint32_t btype,
                                                        uint32_t M, uint32_t N) {
  return (1u << 2) | (1u << 4) | ((atype & 7u) << 7) | ((btype & 7u) << 10) | (0u << 15) |
         (1u << 16) | (((N >> 3) & 0x3Fu) << 17) | (((M >> 4) & 0x1Fu) << 24);
}

}  // namespace sp24
