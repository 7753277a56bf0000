// te_dact_dbias_quantize_noalloc: the activation-gradient + bias-reduction + quantize step for
// callers that cannot allocate device memory when they call it.
//
// Some callers cannot hand this library a workspace: plugin hosts and inference or training
// runtimes that plan every device buffer ahead of time and give an operator no allocator, and
// code on a latency-critical path where cudaMalloc (which synchronizes the whole device) is not
// acceptable.  For them this variant keeps the bias reduction's partial sums in a fixed
// file-scope device array instead of a caller workspace, and allocates nothing.
//
// Properties a caller must know:
//   * The array holds kNoAllocPartials floats (8 MiB).  Every GPU that loads the library keeps
//     it until the process exits.  A call whose reduction needs more (ceil(M / 128) * N_in
//     floats, only when dbias is requested) is rejected with TE_ERR_TOO_LARGE before launching.
//   * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
//     once per device, with that device current).  Make that first call before any stream
//     capture begins on the device.
//   * Every call on a device shares the one array.  Calls that overlap on the GPU (different
//     streams, or host threads without ordering) race on it; order them on one stream.
//   * Nothing in the array has to start at zero: each call writes every partial sum it later
//     reads.  The array keeps the last call's contents.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "te_gb300.h"

namespace te {
namespace {

constexpr size_t kNoAllocPartials = size_t(2) << 20;  // floats: 8 MiB

static __device__ __align__(256) float g_noalloc_partials[kNoAllocPartials];

struct SymbolCache {
  std::mutex mu;
  float* ptr[kMaxDevices] = {};
};

SymbolCache& cache() {
  static SymbolCache c;
  return c;
}

// Device address of g_noalloc_partials on the current device (looked up once per device).
te_status partials_ptr(float** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TE_ERR_UNSUPPORTED;
  SymbolCache& c = cache();
  std::lock_guard<std::mutex> g(c.mu);
  if (!c.ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_partials) != cudaSuccess || p == nullptr)
      return TE_ERR_CUDA;
    c.ptr[dev] = static_cast<float*>(p);
  }
  *out = c.ptr[dev];
  return TE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool enabled(const te_quantizer* q) { return q != nullptr && q->scale != nullptr; }

}  // namespace
}  // namespace te

using namespace te;

extern "C" {

size_t te_dact_dbias_noalloc_capacity(void) { return kNoAllocPartials; }

te_status te_dact_dbias_quantize_noalloc(const void* dy, const void* x_preact, te_dtype dtype,
                                         int64_t M, int64_t N_in, te_act_type act,
                                         const te_quantizer* q, void* dx, te_dtype dx_dtype,
                                         float* dbias, void* stream) {
  if (M < 0 || N_in <= 0 || (dtype != TE_F32 && dtype != TE_BF16) || act < TE_IDENTITY ||
      act > TE_REGLU || dx_dtype < TE_F32 || dx_dtype > TE_E4M3)
    return TE_ERR_INVALID_ARG;
  if (M > 0 && (!dy || (act != TE_IDENTITY && !x_preact) || !dx)) return TE_ERR_INVALID_ARG;
  if (dx_dtype == TE_E4M3 && !enabled(q)) return TE_ERR_INVALID_ARG;
  if (enabled(q) && ((q->mode != TE_SCALING_DELAYED && q->mode != TE_SCALING_CURRENT) ||
                     (q->mode == TE_SCALING_CURRENT && !q->amax) || !aligned4(q->scale) ||
                     !aligned4(q->scale_inv) || !aligned4(q->amax)))
    return TE_ERR_INVALID_ARG;
  const int64_t n_out = is_gated(act) ? N_in / 2 : N_in;
  if ((is_gated(act) && N_in % 2) || n_out % 8) return TE_ERR_UNSUPPORTED;
  if (!aligned16(dy) || !aligned16(x_preact) || !aligned16(dx) || !aligned4(dbias))
    return TE_ERR_UNSUPPORTED;
  if (dbias && M > 0 && dact_dbias_workspace(M, N_in) > kNoAllocPartials * sizeof(float))
    return TE_ERR_TOO_LARGE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dbias && M == 0)
    return cudaMemsetAsync(dbias, 0, size_t(N_in) * 4, s) == cudaSuccess ? TE_OK : TE_ERR_CUDA;
  if (M == 0) return TE_OK;
  float* partials = nullptr;
  if (dbias) {
    te_status st = partials_ptr(&partials);
    if (st != TE_OK) return st;
  }
  // As in te_dact_dbias_quantize, the quantizer only takes part when dx is E4M3.
  const te_quantizer* qq = dx_dtype == TE_E4M3 ? q : nullptr;
  if (qq && qq->amax && cudaMemsetAsync(qq->amax, 0, sizeof(float), s) != cudaSuccess)
    return TE_ERR_CUDA;
  DactArgs a;
  a.dy = dy;
  a.x = x_preact;
  a.dtype = dtype;
  a.M = M;
  a.N_in = N_in;
  a.act = act;
  a.dx = dx;
  a.dbias = dbias;
  a.partials = partials;
  a.cast.out_dtype = dx_dtype;
  if (!enabled(qq)) return launch_dact_dbias(a, s);
  if (qq->mode == TE_SCALING_DELAYED) {
    a.cast.scale = qq->scale;
    a.cast.amax_out = qq->amax;
    a.cast.scale_inv_out = qq->scale_inv;
    return launch_dact_dbias(a, s);
  }
  // Current scaling: the amax pass also reduces dbias; the cast pass only stores dx.
  DactArgs pass1 = a;
  pass1.cast.store = 0;
  pass1.cast.amax_out = qq->amax;
  te_status st = launch_dact_dbias(pass1, s);
  if (st != TE_OK) return st;
  DactArgs pass2 = a;
  pass2.dbias = nullptr;
  pass2.cast.amax_in = qq->amax;
  pass2.cast.scale_out = qq->scale;
  pass2.cast.scale_inv_out = qq->scale_inv;
  return launch_dact_dbias(pass2, s);
}

}  // extern "C"
