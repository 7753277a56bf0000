// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>

#include "te_gb300.h"

namespace te {

// Gated activations take [gate | linear] and apply their base function to the gate half.
__host__ __device__ constexpr bool is_gated(int act) {
  return act == TE_SWIGLU || act == TE_GEGLU || act == TE_REGLU;
}
__host__ __device__ constexpr int gate_act(int act) {
  return act == TE_SWIGLU ? TE_SILU : act == TE_GEGLU ? TE_GELU : act == TE_REGLU ? TE_RELU : act;
}

// Output stage shared by the bandwidth-bound kernels: how fp32 results become the stored
// tensor, and which scalars the kernel reads or writes.
struct CastSpec {
  int out_dtype = TE_BF16;         // TE_F32 / TE_BF16 / TE_E4M3
  int fake_quant = 0;              // quantize then dequantize into out_dtype (F32 / BF16)
  const float* scale = nullptr;    // E4M3 scale to use (delayed scaling)
  const float* amax_in = nullptr;  // current scaling: derive the scale from this amax
  float* amax_out = nullptr;       // atomic max of |pre-cast value| (zeroed by the caller)
  float* scale_out = nullptr;      // written with the scale used (current scaling)
  float* scale_inv_out = nullptr;  // written with 1 / scale
  int store = 1;                   // 0: amax pass of current scaling, nothing stored
};

struct NormFwdArgs {
  const void* x = nullptr;
  int x_dtype = TE_BF16;
  int64_t M = 0, H = 0;
  const void* gamma = nullptr;
  const void* beta = nullptr;
  int norm_type = TE_LAYERNORM;
  int zero_centered_gamma = 0;
  float eps = 1e-6f;
  void* out = nullptr;
  float* mu = nullptr;
  float* rsigma = nullptr;
  CastSpec cast;
  int prefetch = 0;  // rows ahead of the current one each warp asks L2 to fetch (set at launch)
};
te_status launch_norm_fwd(const NormFwdArgs& a, cudaStream_t s);

struct NormBwdArgs {
  const void* dz = nullptr;  // [M, H] upstream gradient, dtype
  const void* x = nullptr;   // [M, H] forward input, dtype
  const float* mu = nullptr;
  const float* rsigma = nullptr;
  const void* gamma = nullptr;
  int dtype = TE_BF16;
  int64_t M = 0, H = 0;
  int norm_type = TE_LAYERNORM;
  int zero_centered_gamma = 0;
  void* dx = nullptr;        // [M, H] dtype
  float* dgamma = nullptr;   // [H]
  float* dbeta = nullptr;    // [H] or null
  float* partials = nullptr; // workspace: [chunks, 2, H]
};
te_status launch_norm_bwd(const NormBwdArgs& a, cudaStream_t s);

// Workspace of te_layernorm_mlp_fwd_host: device staging of x and out plus one forward's.
size_t host_fwd_workspace(int64_t M, int64_t H, int64_t F, int dtype, int act);
size_t norm_bwd_workspace(int64_t M, int64_t H);

struct ActArgs {
  const void* x = nullptr;
  int x_dtype = TE_BF16;
  int64_t M = 0, N_in = 0;
  int act = TE_GELU;
  void* out = nullptr;
  CastSpec cast;
};
te_status launch_act_lu(const ActArgs& a, cudaStream_t s);

struct DactArgs {
  const void* dy = nullptr;
  const void* x = nullptr;
  int dtype = TE_BF16;
  int64_t M = 0, N_in = 0;
  int act = TE_GELU;
  void* dx = nullptr;
  float* dbias = nullptr;
  float* partials = nullptr;  // workspace for the deterministic column reduction
  CastSpec cast;
};
te_status launch_dact_dbias(const DactArgs& a, cudaStream_t s);
size_t dact_dbias_workspace(int64_t M, int64_t N_in);

struct QuantizeArgs {
  const void* x = nullptr;
  int x_dtype = TE_BF16;
  int64_t n = 0;  // elements, multiple of 8
  void* out = nullptr;
  CastSpec cast;
};
te_status launch_quantize(const QuantizeArgs& a, cudaStream_t s);

// dst[C, R] = transpose of src[R, C] (fp32): the tf32 tensor-core path takes K-major operands.
te_status launch_transpose_f32(const float* src, int64_t R, int64_t C, float* dst, cudaStream_t s);

// scale = 448 / amax (the recipe's exceptions included), scale_inv = 1 / scale, for up to
// kMaxScaleUpdates quantizers in one launch.
constexpr int kMaxScaleUpdates = 16;
struct ScaleUpdateArgs {
  int n = 0;
  const float* amax[kMaxScaleUpdates] = {};
  float* scale[kMaxScaleUpdates] = {};
  float* scale_inv[kMaxScaleUpdates] = {};
};
te_status launch_update_scales(const ScaleUpdateArgs& a, cudaStream_t s);

// Tensor-core GEMM D[M, N] = epilogue(alpha * op(A) op(B)).
enum Epilogue { EPI_BIAS = 0, EPI_BIAS_ACT = 1, EPI_BIAS_GATED = 2 };

struct GemmArgs {
  const void* A = nullptr;
  const void* B = nullptr;
  int ab_dtype = TE_BF16;   // TE_BF16 / TE_E4M3 / TE_F32 (tf32)
  int a_kmajor = 1;         // A stored [M, K] (1) or [K, M] (0)
  int b_kmajor = 0;         // B stored [N, K] (1) or [K, N] (0)
  int64_t M = 0, N = 0, K = 0;  // N = accumulator columns; gated: N = 2F
  const float* a_scale_inv = nullptr;
  const float* b_scale_inv = nullptr;
  int epilogue = EPI_BIAS;
  int act = TE_IDENTITY;
  const void* bias = nullptr;   // [N]
  int bias_dtype = TE_F32;
  int h_dtype = TE_F32;         // dtype the pre-activation is rounded to (act epilogues)
  void* saved_h = nullptr;      // [M, N] pre-activation, h_dtype
  void* D = nullptr;            // [M, N] or [M, N/2] gated
  CastSpec cast;                // output stage of D (amax / E4M3 of the activation)
  // Optional scratch (256-byte aligned) for splitting the last wave's tiles along K; without it
  // no tile is split.
  void* split_ws = nullptr;
  size_t split_ws_bytes = 0;
};
te_status launch_gemm(const GemmArgs& g, cudaStream_t s);
// Bytes of split_ws that launch_gemm would use for this GEMM on the current device (0: none).
size_t gemm_split_workspace(int64_t M, int64_t N, int64_t K, int ab_dtype, int epilogue);

// Device status word (TE_OK or the first failure a kernel recorded).
int* device_status_ptr();
te_status read_and_clear_device_status(int32_t* out);

int num_sms();

// The streaming reference of te_stream_probe (n_out 16-byte vectors written, each from `ratio`
// read; n_out = 0: n_read vectors read only).
te_status launch_stream_probe(const uint4* src, uint4* dst, size_t n_out, int ratio,
                              size_t n_read, cudaStream_t s);

// Launches `kernel` as a programmatic dependent of the work queued before it on `s`: its launch
// may overlap the previous kernel's tail once every CTA of that kernel has executed
// griddepcontrol.launch_dependents (or exited), and the kernel itself executes
// griddepcontrol.wait before it reads anything the previous kernel wrote.
template <typename... KArgs, typename... Args>
te_status launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, cudaStream_t s,
                           Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...) == cudaSuccess ? TE_OK
                                                                                     : TE_ERR_CUDA;
}

// A value set up once per device and shared by every host thread: get() runs make(&value) for
// the current device the first time (make returns false on failure, and is then retried on the
// next call) and returns the cached value afterwards.  Devices numbered kMaxDevices or above
// are set up on every call, uncached.
constexpr int kMaxDevices = 64;
template <typename T>
class PerDevice {
 public:
  template <class Make>
  bool get(T* out, Make&& make) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (dev < 0 || dev >= kMaxDevices) return make(out);
    std::lock_guard<std::mutex> lock(mu_);
    if (!have_[dev]) {
      if (!make(&value_[dev])) return false;
      have_[dev] = true;
    }
    *out = value_[dev];
    return true;
  }

 private:
  std::mutex mu_;
  T value_[kMaxDevices] = {};
  bool have_[kMaxDevices] = {};
};

// 2-D TMA tensor map over a row-major [outer, inner] matrix of dtype, boxes of
// box_inner x box_outer elements, 128-byte swizzle or none, out-of-bounds reads zero.
bool make_tmap_2d(CUtensorMap* tm, const void* ptr, int dtype, uint64_t inner, uint64_t outer,
                  uint32_t box_inner, uint32_t box_outer, bool swizzle128);

// Brackets one kernel launch with profiling events when te_profile_begin is active.
class ProfileScope {
 public:
  ProfileScope(int kind, cudaStream_t stream);
  ~ProfileScope();
  ProfileScope(const ProfileScope&) = delete;
  ProfileScope& operator=(const ProfileScope&) = delete;

 private:
  int kind_;
  cudaStream_t stream_;
  int slot_ = -1;
};

}  // namespace te
