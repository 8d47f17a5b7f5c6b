// Inline-PTX building blocks for sm_103a: mbarriers with bounded waits, TMA tiled loads,
// tcgen05 (TMEM allocation, MMA, commit, TMEM loads/stores) and shared-memory descriptors.
//
// Every wait here is bounded: it polls with mbarrier.try_wait and gives up after a wall-clock
// budget read from %globaltimer, so that a logic error ends the kernel with an error status
// instead of leaving the GPU spinning.
#pragma once
#include <cstdint>
#include <cuda.h>

namespace usp {

constexpr uint32_t kErrTimeout = 1u;  // bit set in the status word when a bounded wait gives up

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// mbarrier operations on a shared-memory address (the pointer forms convert theirs).
__device__ __forceinline__ void mbar_arrive_at(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) { mbar_arrive_at(smem_u32(bar)); }

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_at(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  return mbar_try_wait_at(smem_u32(bar), parity);
}

// Bounded wait for the phase with the given parity.  Returns false if the budget ran out or if
// *abort became non-zero (another role gave up); on a timeout it sets *abort and ORs kErrTimeout
// into *status.
__device__ __forceinline__ bool mbar_wait_at(uint32_t bar, uint32_t parity, volatile int* abort,
                                             uint32_t* status, uint64_t budget_ns) {
  if (mbar_try_wait_at(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_at(bar, parity)) return true;
    if ((it & 63u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > budget_ns) {
        *abort = 1;
        if (status) atomicOr(status, kErrTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint32_t* status, uint64_t budget_ns) {
  return mbar_wait_at(smem_u32(bar), parity, abort, status, budget_ns);
}

// Wait used only while draining at exit: bounded, ignores the abort flag.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
  uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > budget_ns) return;
  }
}

// 4-D tiled load {c0, c1, c2, c3} -> shared memory, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// 5-D tiled load {c0, c1, c2, c3, c4} -> shared memory, completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_5d(void* smem_dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, int c4, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_u32(bar))
      : "memory");
}

// Programmatic dependent launch, kernel side: let the next kernel of the stream be scheduled once
// every CTA of this one has started, then wait until the previous kernel has completed and its
// memory is visible (a no-op when the kernel was launched without the programmatic attribute).
// Call before the kernel's first global memory access.
__device__ __forceinline__ void pdl_prologue() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The two halves of pdl_prologue(), for kernels that compute their first addresses from the
// parameters before waiting: launch_dependents at the start, wait before the first global memory
// access (load or store).
// A kernel launched this way reads the previous kernel's outputs with coherent loads only (plain
// or ld.global.cs), never ld.global.nc (__ldg): a non-coherent load declares its data constant for
// the whole kernel, which does not hold before the wait returns, and such a load may then be
// scheduled ahead of the wait.  (Observed: a merge whose LSE loads were ld.global.nc read the
// previous round's LSE when it followed, back to back, the copy that wrote them.)
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------------------------
// tcgen05
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
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

// The MMA groups and the commit below are warp-wide: all 32 lanes of a converged warp execute
// them with the same operands, and the lane `elect.sync` picks issues the tcgen05 instructions.
// Running the issuing role on a whole warp keeps its loop state and descriptors warp-uniform.

// S = A B^T over K = 128 (the 8 K-steps of a 128x128 score tile), issued as one block:
// a_lo / b_lo are the low descriptor words of the K-step-0 operands (start address >> 4 | LBO field),
// hi the shared high word; K-step kk adds (kk / 4) * 1024 + (kk % 4) * 2 (16-byte units) to both.
__device__ __forceinline__ void mma_group_qk8(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                              uint32_t hi, uint32_t idesc) {
  asm volatile("{\n\t.reg .pred ee;\n\telect.sync _|ee, 0xffffffff;\n\t.reg .pred pz, pa;\n\t.reg .b32 alo, blo;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 pz, 0, 0;\n\tsetp.eq.b32 pa, 0, 0;\n\tadd.u32 alo, %1, 0;\n\tadd.u32 blo, %2, 0;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pz;\n\tadd.u32 alo, %1, 2;\n\tadd.u32 blo, %2, 2;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 4;\n\tadd.u32 blo, %2, 4;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 6;\n\tadd.u32 blo, %2, 6;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 1024;\n\tadd.u32 blo, %2, 1024;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 1026;\n\tadd.u32 blo, %2, 1026;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 1028;\n\tadd.u32 blo, %2, 1028;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 1030;\n\tadd.u32 blo, %2, 1030;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\t}" ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc) : "memory");
}

// S = A B^T over K = 64 (the 4 K-steps of a 128x128 score tile), issued as one block:
// a_lo / b_lo are the low descriptor words of the K-step-0 operands (start address >> 4 | LBO field),
// hi the shared high word; K-step kk adds (kk / 4) * 1024 + (kk % 4) * 2 (16-byte units) to both.
__device__ __forceinline__ void mma_group_qk4(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                              uint32_t hi, uint32_t idesc) {
  asm volatile("{\n\t.reg .pred ee;\n\telect.sync _|ee, 0xffffffff;\n\t.reg .pred pz, pa;\n\t.reg .b32 alo, blo;\n\t.reg .b64 da, db;\n\tsetp.ne.b32 pz, 0, 0;\n\tsetp.eq.b32 pa, 0, 0;\n\tadd.u32 alo, %1, 0;\n\tadd.u32 blo, %2, 0;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pz;\n\tadd.u32 alo, %1, 2;\n\tadd.u32 blo, %2, 2;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 4;\n\tadd.u32 blo, %2, 4;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\tadd.u32 alo, %1, 6;\n\tadd.u32 blo, %2, 6;\n\tmov.b64 da, {alo, %3};\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %4, pa;\n\t}" ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(hi), "r"(idesc) : "memory");
}

// O (+)= P V over the 128 keys of a tile, issued as one block: P from TMEM (keys 2c, 2c+1 packed
// in column p_tmem + c, c < 64), V from shared memory (MN-major, K-step kk adds kk * 128 in
// 16-byte units to b_lo); the first K-step accumulates iff acc_first != 0.
__device__ __forceinline__ void mma_group_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t b_lo,
                                             uint32_t hi, uint32_t idesc, uint32_t acc_first) {
  asm volatile("{\n\t.reg .pred ee;\n\telect.sync _|ee, 0xffffffff;\n\t.reg .pred pf, pa;\n\t.reg .b32 alo, blo;\n\t.reg .b64 db;\n\tsetp.ne.b32 pf, %5, 0;\n\tsetp.eq.b32 pa, 0, 0;\n\tadd.u32 alo, %1, 0;\n\tadd.u32 blo, %2, 0;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pf;\n\tadd.u32 alo, %1, 8;\n\tadd.u32 blo, %2, 128;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\tadd.u32 alo, %1, 16;\n\tadd.u32 blo, %2, 256;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\tadd.u32 alo, %1, 24;\n\tadd.u32 blo, %2, 384;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\tadd.u32 alo, %1, 32;\n\tadd.u32 blo, %2, 512;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\tadd.u32 alo, %1, 40;\n\tadd.u32 blo, %2, 640;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\tadd.u32 alo, %1, 48;\n\tadd.u32 blo, %2, 768;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\tadd.u32 alo, %1, 56;\n\tadd.u32 blo, %2, 896;\n\tmov.b64 db, {blo, %3};\n\t@ee tcgen05.mma.cta_group::1.kind::f16 [%0], [alo], db, %4, pa;\n\t}" ::"r"(d_tmem), "r"(p_tmem), "r"(b_lo), "r"(hi), "r"(idesc),
               "r"(acc_first)
               : "memory");
}

// Arrive once on `bar` (from the elected lane) when every tcgen05 operation the warp's issuing
// lane issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred ee;\n\telect.sync _|ee, 0xffffffff;\n\t@ee tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16-lane TMEM accesses.  Thread t of a warp holds, per repetition k, for lanes base + t/4 and
// base + t/4 + 8: .16x256b -> columns 8k + 2(t%4) + {0, 1} (registers 4k, 4k+1 for the first lane,
// 4k+2, 4k+3 for the second); .16x128b -> column 4k + t%4 (registers 2k, 2k+1).
__device__ __forceinline__ void tmem_ld_16x256b_x16(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st_16x256b_x16(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
               : "memory");
}
__device__ __forceinline__ void tmem_st_16x256b_x8(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
               : "memory");
}
__device__ __forceinline__ void tmem_st_16x128b_x4(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x4.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_16x128b_x8(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.16x128b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};"
               :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (0 = K), bit 16 B major (1 = MN), bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (b_mn_major << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// ---------------------------------------------------------------------------------------------
// Special-function-unit instructions (PTX instructions, not library routines)
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two floats to bf16x2 (round to nearest even): `lo` in bits 0-15, `hi` in bits 16-31.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// ---------------------------------------------------------------------------------------------
// Packed fp32x2 arithmetic (sm_100+): two lanes of work per instruction.
// ---------------------------------------------------------------------------------------------
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Register rebalancing between warpgroups (all threads of a warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

}  // namespace usp
