// tdt_async.cuh -- asynchronous copies and mbarriers (PTX ISA: cp.async,
// mbarrier) used by the lattice kernels.
#pragma once

#include "tdt_common.cuh"

namespace tdt {

__device__ __forceinline__ unsigned smem_u32(const void *p) {
  return (unsigned)__cvta_generic_to_shared(p);
}

// 16-byte copy global -> shared (cp.async, L2 only), grouped per thread.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}
// The same if `pred` (predicated, no branch).
__device__ __forceinline__ void cp_async16_if(bool pred, void *smem, const void *gmem) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t"
      "@p cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(smem_u32(smem)),
      "l"(gmem), "r"((int)pred));
}
// 8-byte copy global -> shared if `pred` (cp.async.ca: may allocate in L1,
// which is invalidated at every kernel launch; each address is copied once).
// Predicated rather than branched around, so that a warp in which one lane
// copies does not diverge.
__device__ __forceinline__ void cp_async8_if(bool pred, void *smem, const void *gmem) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t"
      "@p cp.async.ca.shared.global [%0], [%1], 8;\n\t}" ::"r"(smem_u32(smem)),
      "l"(gmem), "r"((int)pred));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
// Makes mbarrier initialisations visible to the other threads and to the
// other CTAs of a cluster.
__device__ __forceinline__ void fence_mbar_init_cluster() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Arrive on a local mbarrier and expect `bytes` more transaction bytes this phase.
__device__ __forceinline__ void arrive_expect_tx(unsigned long long *bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
// Non-blocking probe of a phase (test_wait never suspends the thread, so a
// completion signalled from another SM is seen at the next probe).
__device__ __forceinline__ bool test_wait_parity(unsigned long long *bar, unsigned parity) {
  unsigned ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// About one second at the GB300 clock: far beyond any legitimate wait.
constexpr long long kWaitLimitCycles = 2000000000LL;
// Wait for the completion of the phase of parity `parity` for at most
// `limit` clock cycles; false on timeout.
__device__ __forceinline__ bool wait_parity_bounded(unsigned long long *bar, unsigned parity,
                                                    long long limit) {
  if (test_wait_parity(bar, parity)) return true;
  const long long t0 = clock64();
  while (!test_wait_parity(bar, parity))
    if (clock64() - t0 > limit) return false;
  return true;
}

}  // namespace tdt
