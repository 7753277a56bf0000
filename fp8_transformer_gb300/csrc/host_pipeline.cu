// Forward of the LayerNorm MLP block with the activations in host memory (serving from host
// buffers; no counterpart on the pages beyond the forward itself).
//
// The rows are cut into `chunks` slices (see slice_rows).  Every host -> device copy is issued
// at once on a copy-in stream the library keeps per device; the forward of slice c runs on the
// caller's stream as soon as slice c has landed, and its result goes back on a copy-out stream the
// moment it is computed.  So slice c + 1 crosses the host link while slice c computes and
// slice c - 1 returns: only the first slice's copy in and the last slice's copy out are not
// hidden behind tensor-core work.  The caller's stream finally waits for the last copy out, so
// the call is as asynchronous, and as ordered, as every other call on that stream.
#include <mutex>

#include "kernels.h"

namespace te {
namespace {

constexpr int kMaxChunks = 16;

struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t landed[kMaxChunks] = {};
  cudaEvent_t computed[kMaxChunks] = {};
};

HostPipe g_pipes[64];
std::mutex g_pipes_mu;

// The current device's copy streams and events, created on first use.
te_status host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return TE_ERR_CUDA;
  if (dev < 0 || dev >= 64) return TE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_pipes_mu);
  HostPipe& p = g_pipes[dev];
  if (!p.ready) {
    const unsigned f = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, f) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.done, f) != cudaSuccess)
      return TE_ERR_CUDA;
    for (int c = 0; c < kMaxChunks; ++c)
      if (cudaEventCreateWithFlags(&p.landed[c], f) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.computed[c], f) != cudaSuccess)
        return TE_ERR_CUDA;
    p.ready = true;
  }
  *out = &p;
  return TE_OK;
}

size_t align256(size_t b) { return (b + 255) / 256 * 256; }

// Row counts of the slices.  Only the first slice's copy in and the last slice's copy out are
// not hidden behind compute, so the two edge slices are small; the middle ones are large,
// where the GEMMs fill the SM pairs (one edge slice weighs 1, a middle one 7).  Every slice but
// the last is a multiple of 256 rows, the height of an SM-pair GEMM tile.
int slice_rows(int64_t M, int chunks, int64_t (&rows)[kMaxChunks]) {
  if (chunks == 1 || M <= 256) {
    rows[0] = M;
    return 1;
  }
  const int64_t weight = chunks == 2 ? 2 : 2 + 7 * int64_t(chunks - 2);
  int n = 0;
  int64_t left = M;
  for (int c = 0; c < chunks && left > 0; ++c) {
    const int64_t w = (c == 0 || c == chunks - 1) ? 1 : 7;
    int64_t r = (M * w / weight + 255) / 256 * 256;
    if (r < 256) r = 256;
    if (c == chunks - 1 || r > left) r = left;
    rows[n++] = r;
    left -= r;
  }
  if (left > 0) rows[n - 1] += left;
  return n;
}

}  // namespace

size_t host_fwd_workspace(int64_t M, int64_t H, int64_t F, int dtype, int act) {
  const size_t stage = align256(size_t(M) * H * (dtype == TE_F32 ? 4 : 2));
  return 2 * stage + te_workspace_size(TE_OP_LAYERNORM_MLP_FWD, M, H, F, te_dtype(dtype), 0,
                                       te_dtype(dtype), te_act_type(act));
}

}  // namespace te

using namespace te;

extern "C" te_status te_layernorm_mlp_fwd_host(
    const void* x_host, const void* gamma, const void* beta, const void* kernel1,
    const void* kernel2, const void* bias1, const void* bias2, te_norm_type norm_type,
    int zero_centered_gamma, float epsilon, te_act_type act, int64_t M, int64_t H, int64_t F,
    te_dtype dtype, void* out_host, int chunks, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || H <= 0 || F <= 0 || chunks < 1 || chunks > kMaxChunks ||
      (dtype != TE_BF16 && dtype != TE_F32))
    return TE_ERR_INVALID_ARG;
  if (M > 0 && (!x_host || !out_host)) return TE_ERR_INVALID_ARG;
  if (M == 0) return TE_OK;
  if (!workspace || ws_bytes < host_fwd_workspace(M, H, F, dtype, act)) return TE_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 255u) return TE_ERR_UNSUPPORTED;
  HostPipe* p = nullptr;
  te_status st = host_pipe(&p);
  if (st != TE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t esz = dtype == TE_F32 ? 4 : 2;
  const size_t row_bytes = size_t(H) * esz;
  const size_t stage = align256(size_t(M) * row_bytes);
  char* x_dev = static_cast<char*>(workspace);
  char* out_dev = x_dev + stage;
  void* fwd_ws = out_dev + stage;
  const size_t fwd_bytes = ws_bytes - 2 * stage;
  int64_t rows[kMaxChunks], first[kMaxChunks];
  const int n = slice_rows(M, chunks, rows);
  for (int64_t c = 0, r = 0; c < n; r += rows[c], ++c) first[c] = r;
  // the copies start only after the work already queued on the caller's stream
  if (cudaEventRecord(p->start, s) != cudaSuccess || cudaStreamWaitEvent(p->in, p->start, 0) ||
      cudaStreamWaitEvent(p->out, p->start, 0))
    return TE_ERR_CUDA;
  for (int c = 0; c < n; ++c) {
    const int64_t r0 = first[c], m = rows[c];
    if (cudaMemcpyAsync(x_dev + r0 * row_bytes, static_cast<const char*>(x_host) + r0 * row_bytes,
                        size_t(m) * row_bytes, cudaMemcpyHostToDevice, p->in) != cudaSuccess ||
        cudaEventRecord(p->landed[c], p->in) != cudaSuccess)
      return TE_ERR_CUDA;
  }
  for (int c = 0; c < n; ++c) {
    const int64_t r0 = first[c], m = rows[c];
    if (cudaStreamWaitEvent(s, p->landed[c], 0) != cudaSuccess) return TE_ERR_CUDA;
    st = te_layernorm_mlp_fwd(x_dev + r0 * row_bytes, gamma, beta, kernel1, kernel2, dtype, bias1,
                              bias2, norm_type, zero_centered_gamma, epsilon, act, nullptr, m, H, F,
                              dtype, out_dev + r0 * row_bytes, nullptr, nullptr, nullptr, nullptr, nullptr,
                              fwd_ws, fwd_bytes, stream);
    if (st != TE_OK) return st;
    if (cudaEventRecord(p->computed[c], s) != cudaSuccess ||
        cudaStreamWaitEvent(p->out, p->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(static_cast<char*>(out_host) + r0 * row_bytes, out_dev + r0 * row_bytes,
                        size_t(m) * row_bytes, cudaMemcpyDeviceToHost, p->out) != cudaSuccess)
      return TE_ERR_CUDA;
  }
  if (cudaEventRecord(p->done, p->out) != cudaSuccess || cudaStreamWaitEvent(s, p->done, 0))
    return TE_ERR_CUDA;
  return TE_OK;
}
