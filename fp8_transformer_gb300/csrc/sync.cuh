// mbarrier / bulk-copy wrappers (inline PTX, sm_90+ forms used on sm_103a) and the bounded
// wait every spin on an mbarrier goes through.
#pragma once

#include <stdint.h>

#include "te_gb300.h"

namespace te {

constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: a pipeline wait that gives up
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s: waiting for own copies in flight

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes initialized barriers visible to the async proxy (TMA / bulk copies).
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with parity `parity`.  Returns false without waiting further
// when `abort_flag` (may be null) is raised and check_abort is set, or when `limit_ns` passes;
// the latter records TE_ERR_TIMEOUT in *status (first failure wins) and raises the flag.
static __device__ __noinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                          int* status, uint64_t limit_ns, bool check_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31) == 0) {
      if (check_abort && abort_flag && *abort_flag) return false;
      if (global_ns() - t0 > limit_ns) {
        if (status) atomicCAS(status, 0, int(TE_ERR_TIMEOUT));
        if (abort_flag) *abort_flag = 1;
        return false;
      }
    }
  }
}

// One contiguous global -> shared copy by the bulk-copy (TMA) engine, completing on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Asks the bulk-copy engine to bring `bytes` of global memory at `src` into L2 (no data returns
// to the SM, nothing to wait for).  src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// One 2-D TMA tile load into this CTA's shared memory, completing on `bar` (this CTA).
// c0 is the inner (contiguous) coordinate in elements, c1 the row.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// Orders earlier generic-proxy accesses of shared memory before later async-proxy writes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace te
