// Self-test of the bounded-wait path (no counterpart on the pages; it checks this library's own
// failure reporting).  One thread waits on an mbarrier that nothing completes, with a short
// limit: the wait gives up, records TE_ERR_TIMEOUT in the device status word and returns, the
// kernel exits normally and the context stays usable.  This is the same wait, with the same
// bookkeeping, that every pipeline of the GEMM and the norm backward goes through.
#include "kernels.h"
#include "sync.cuh"

namespace te {
namespace {

__global__ void wait_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    mbar_init_fence();
  }
  __syncthreads();
  // phase 0 of a fresh barrier with one expected arrival and no arriving thread: never completes
  if (threadIdx.x == 0) wait_bounded(smem_u32(&bar), 0, nullptr, status, limit_ns, false);
}

}  // namespace
}  // namespace te

extern "C" te_status te_selftest_wait_timeout(int64_t limit_us, void* stream) {
  if (limit_us <= 0 || limit_us > 1000000) return TE_ERR_INVALID_ARG;
  te::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      te::device_status_ptr(), uint64_t(limit_us) * 1000u);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}
