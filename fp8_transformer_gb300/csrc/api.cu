// C ABI of the fused norm + feed-forward block: argument validation, workspace carving and
// the composition of the kernels on the caller's stream.  Declarations and the contract of
// every entry point are in include/te_gb300.h.
#include <cuda_runtime.h>

#include <cstdint>
#include <initializer_list>
#include <utility>

#include "kernels.h"
#include "te_gb300.h"

namespace te {
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool opt_aligned16(const void* p) { return p == nullptr || aligned16(p); }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

size_t esize(int dt) { return dt == TE_F32 ? 4 : dt == TE_BF16 ? 2 : 1; }
bool is_act_dtype(int dt) { return dt == TE_F32 || dt == TE_BF16; }
bool valid_act(int a) { return a >= TE_IDENTITY && a <= TE_REGLU; }
bool enabled(const te_quantizer* q) { return q != nullptr && q->scale != nullptr; }

bool quantizer_ok(const te_quantizer* q) {
  if (!enabled(q)) return true;
  if (!aligned4(q->scale) || !aligned4(q->scale_inv) || !aligned4(q->amax)) return false;
  if (q->mode != TE_SCALING_DELAYED && q->mode != TE_SCALING_CURRENT) return false;
  // Current scaling keeps this call's amax between its two passes.
  if (q->mode == TE_SCALING_CURRENT && q->amax == nullptr) return false;
  return true;
}

constexpr size_t kAlign = 256;
size_t round_up(size_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

// Sequential carving of the caller's workspace into 256-byte aligned regions.
struct Carver {
  uint8_t* base;
  size_t used = 0;
  explicit Carver(void* b) : base(static_cast<uint8_t*>(b)) {}
  void* take(size_t bytes) {
    void* p = base ? base + used : nullptr;
    used += round_up(bytes);
    return p;
  }
};

// The scratch for splitting GEMM tails along K (launch_gemm) is carved last: a workspace that
// stops short of it still serves the call, with no tile split.  The GEMMs of one call run one
// after another on its stream, so they share the region, sized for the largest.
struct SplitScratch {
  size_t offset = 0;  // where the region starts in the workspace
  size_t required = 0;  // workspace bytes the call needs (everything before the region)
};

SplitScratch carve_split(Carver& c, std::initializer_list<size_t> needs) {
  SplitScratch r;
  r.required = c.used;
  r.offset = c.used;
  size_t most = 0;
  for (size_t n : needs) most = n > most ? n : most;
  if (most) c.take(most);
  return r;
}

void give_split(GemmArgs& g, const SplitScratch& sc, void* ws, size_t ws_bytes) {
  if (ws && ws_bytes > sc.offset) {
    g.split_ws = static_cast<uint8_t*>(ws) + sc.offset;
    g.split_ws_bytes = ws_bytes - sc.offset;
  }
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

te_status zero_scalar(float* p, cudaStream_t s) {
  if (!p) return TE_OK;
  return cudaMemsetAsync(p, 0, sizeof(float), s) == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

// Runs a bandwidth-bound producer once (no quantizer, or delayed scaling) or twice (current
// scaling: an amax pass that stores nothing, then the cast pass with scale = 448 / amax).
template <class Launch>
te_status run_cast(const te_quantizer* q, int out_dtype, int fake_quant, cudaStream_t s,
                   Launch&& launch) {
  CastSpec c;
  c.out_dtype = out_dtype;
  c.fake_quant = fake_quant;
  if (q) {
    te_status st = zero_scalar(q->amax, s);
    if (st != TE_OK) return st;
  }
  if (!enabled(q)) {
    c.amax_out = q ? q->amax : nullptr;
    return launch(c);
  }
  if (q->mode == TE_SCALING_DELAYED) {
    c.scale = q->scale;
    c.amax_out = q->amax;
    c.scale_inv_out = q->scale_inv;
    return launch(c);
  }
  CastSpec pass1 = c;
  pass1.store = 0;
  pass1.amax_out = q->amax;
  te_status st = launch(pass1);
  if (st != TE_OK) return st;
  CastSpec pass2 = c;
  pass2.amax_in = q->amax;
  pass2.scale_out = q->scale;
  pass2.scale_inv_out = q->scale_inv;
  return launch(pass2);
}

// Workspace layout of the composed forward passes (shared by te_workspace_size and the calls).
struct FwdLayout {
  void* ln = nullptr;     // normalized output (when not saved by the caller)
  void* kt1 = nullptr;    // fp32: kernel1 / the dense kernel transposed to [out, in]
  void* kt2 = nullptr;    // fp32: kernel2 transposed
  void* kq1 = nullptr;    // E4M3 copy of kernel1 / the dense kernel
  void* kq2 = nullptr;    // E4M3 copy of kernel2
  void* a2 = nullptr;     // activation output, GEMM2 operand
  void* a2_hi = nullptr;  // fp32 activation output awaiting its current-scaling cast
  SplitScratch split;
  size_t bytes = 0;
};

FwdLayout dense_layout(void* ws, int64_t M, int64_t H, int64_t N, int dtype, bool quant,
                       int kernel_dtype, bool have_saved_ln) {
  Carver c(ws);
  FwdLayout L;
  if (!have_saved_ln) L.ln = c.take(size_t(M) * H * (quant ? 1 : esize(dtype)));
  if (quant && kernel_dtype != TE_E4M3) L.kq1 = c.take(size_t(H) * N);
  if (!quant && dtype == TE_F32) L.kt1 = c.take(size_t(H) * N * 4);
  L.split = carve_split(c, {gemm_split_workspace(M, N, H, quant ? TE_E4M3 : dtype, EPI_BIAS)});
  L.bytes = c.used;
  return L;
}

FwdLayout mlp_layout(void* ws, int64_t M, int64_t H, int64_t F, int dtype, bool quant,
                     int kernel_dtype, int act, bool have_saved_ln) {
  Carver c(ws);
  FwdLayout L;
  const int64_t F1 = is_gated(act) ? 2 * F : F;
  if (!have_saved_ln) L.ln = c.take(size_t(M) * H * (quant ? 1 : esize(dtype)));
  L.a2 = c.take(size_t(M) * F * (quant ? 1 : esize(dtype)));
  if (quant) {
    L.a2_hi = c.take(size_t(M) * F * 4);  // fp32: cast once, from the fp32 activation
    if (kernel_dtype != TE_E4M3) {
      L.kq1 = c.take(size_t(H) * F1);
      L.kq2 = c.take(size_t(F) * H);
    }
  } else if (dtype == TE_F32) {
    L.kt1 = c.take(size_t(H) * F1 * 4);
    L.kt2 = c.take(size_t(F) * H * 4);
  }
  const int gd = quant ? TE_E4M3 : dtype;
  L.split = carve_split(c, {gemm_split_workspace(M, F1, H, gd, is_gated(act) ? EPI_BIAS_GATED : EPI_BIAS_ACT),
                            gemm_split_workspace(M, H, F, gd, EPI_BIAS)});
  L.bytes = c.used;
  return L;
}

// Workspace of te_layernorm_mlp_bwd.  The three reductions run one after another on the
// stream, so they share one partial-sum region.
struct BwdLayout {
  void* partials = nullptr;
  void* a = nullptr;     // recomputed activation [M, F], dtype
  void* da = nullptr;    // [M, F], dtype
  void* dh = nullptr;    // [M, F'], E4M3 or dtype
  void* dln = nullptr;   // [M, H], dtype
  void* kq1 = nullptr;   // E4M3 kernel1 when quantized here
  SplitScratch split;
  size_t bytes = 0;
};

BwdLayout bwd_layout(void* ws, int64_t M, int64_t H, int64_t F, int dtype, bool quant,
                     int kernel_dtype, int act) {
  Carver c(ws);
  BwdLayout L;
  const int64_t F1 = is_gated(act) ? 2 * F : F;
  size_t part = dact_dbias_workspace(M, H);
  if (dact_dbias_workspace(M, F1) > part) part = dact_dbias_workspace(M, F1);
  if (norm_bwd_workspace(M, H) > part) part = norm_bwd_workspace(M, H);
  L.partials = c.take(part);
  L.a = c.take(size_t(M) * F * esize(dtype));
  L.da = c.take(size_t(M) * F * esize(dtype));
  L.dh = c.take(size_t(M) * F1 * (quant ? 1 : esize(dtype)));
  L.dln = c.take(size_t(M) * H * esize(dtype));
  if (quant && kernel_dtype != TE_E4M3) L.kq1 = c.take(size_t(H) * F1);
  const int gd = quant ? TE_E4M3 : dtype;
  L.split = carve_split(c, {gemm_split_workspace(F, H, M, dtype, EPI_BIAS),
                            gemm_split_workspace(M, F, H, dtype, EPI_BIAS),
                            gemm_split_workspace(M, H, F1, gd, EPI_BIAS),
                            gemm_split_workspace(H, F1, M, gd, EPI_BIAS)});
  L.bytes = c.used;
  return L;
}

// Workspace of te_layernorm_dense_bwd (reductions run one after another, so they share one
// partials buffer).
struct DenseBwdLayout {
  void* partials = nullptr;
  void* dyq = nullptr;  // E4M3 dy (FP8 mode)
  void* kq = nullptr;   // E4M3 kernel when quantized here
  void* dln = nullptr;  // [M, H], dtype
  SplitScratch split;
  size_t bytes = 0;
};

DenseBwdLayout dense_bwd_layout(void* ws, int64_t M, int64_t H, int64_t N, int dtype, bool quant,
                                int kernel_dtype) {
  Carver c(ws);
  DenseBwdLayout L;
  size_t part = dact_dbias_workspace(M, N);
  if (norm_bwd_workspace(M, H) > part) part = norm_bwd_workspace(M, H);
  L.partials = c.take(part);
  if (quant) L.dyq = c.take(size_t(M) * N);
  if (quant && kernel_dtype != TE_E4M3) L.kq = c.take(size_t(H) * N);
  L.dln = c.take(size_t(M) * H * esize(dtype));
  const int gd = quant ? TE_E4M3 : dtype;
  L.split = carve_split(c, {gemm_split_workspace(M, H, N, gd, EPI_BIAS),
                            gemm_split_workspace(H, N, M, gd, EPI_BIAS)});
  L.bytes = c.used;
  return L;
}

te_status norm_into(const void* x, int dtype, int64_t M, int64_t H, const void* gamma,
                    const void* beta, int norm_type, int zcg, float eps, const te_quantizer* q,
                    void* out, int out_dtype, float* mu, float* rsigma, cudaStream_t s) {
  return run_cast(out_dtype == TE_E4M3 ? q : nullptr, out_dtype, 0, s, [&](const CastSpec& c) {
    NormFwdArgs a;
    a.x = x;
    a.x_dtype = dtype;
    a.M = M;
    a.H = H;
    a.gamma = gamma;
    a.beta = beta;
    a.norm_type = norm_type;
    a.zero_centered_gamma = zcg;
    a.eps = eps;
    a.out = out;
    a.mu = mu;
    a.rsigma = rsigma;
    a.cast = c;
    if (out_dtype != TE_E4M3 && q) a.cast.amax_out = q->amax;
    return launch_norm_fwd(a, s);
  });
}

te_status quantize_into(const void* x, int dtype, int64_t n, const te_quantizer* q, void* out,
                        cudaStream_t s) {
  return run_cast(q, TE_E4M3, 0, s, [&](const CastSpec& c) {
    QuantizeArgs a;
    a.x = x;
    a.x_dtype = dtype;
    a.n = n;
    a.out = out;
    a.cast = c;
    return launch_quantize(a, s);
  });
}

}  // namespace
}  // namespace te

using namespace te;

extern "C" {

const char* te_status_string(te_status status) {
  switch (status) {
    case TE_OK: return "TE_OK";
    case TE_ERR_INVALID_ARG: return "TE_ERR_INVALID_ARG: invalid argument";
    case TE_ERR_UNSUPPORTED: return "TE_ERR_UNSUPPORTED: shape, alignment or dtype not supported";
    case TE_ERR_CUDA: return "TE_ERR_CUDA: CUDA runtime error";
    case TE_ERR_TIMEOUT: return "TE_ERR_TIMEOUT: a device pipeline wait timed out";
    case TE_ERR_WORKSPACE: return "TE_ERR_WORKSPACE: workspace missing or too small";
    case TE_ERR_TOO_LARGE:
      return "TE_ERR_TOO_LARGE: problem exceeds the fixed scratch of the no-allocation entry point";
  }
  return "unknown te_status";
}

int te_version(void) { return 200; }

te_status te_get_device_status(int32_t* device_status) {
  return read_and_clear_device_status(device_status);
}

size_t te_workspace_size(te_op op, int64_t M, int64_t H, int64_t F_or_N, te_dtype dtype,
                         int quantized, te_dtype kernel_dtype, te_act_type act) {
  switch (op) {
    case TE_OP_DACT_DBIAS: return dact_dbias_workspace(M, F_or_N);
    case TE_OP_NORM_BWD: return norm_bwd_workspace(M, H);
    case TE_OP_LAYERNORM_DENSE_FWD:
      return dense_layout(nullptr, M, H, F_or_N, dtype, quantized != 0, kernel_dtype, false).bytes;
    case TE_OP_LAYERNORM_MLP_FWD:
      return mlp_layout(nullptr, M, H, F_or_N, dtype, quantized != 0, kernel_dtype, act, false).bytes;
    case TE_OP_LAYERNORM_MLP_BWD:
      return bwd_layout(nullptr, M, H, F_or_N, dtype, quantized != 0, kernel_dtype, act).bytes;
    case TE_OP_LAYERNORM_MLP_FWD_HOST:
      return host_fwd_workspace(M, H, F_or_N, dtype, act);
    case TE_OP_GEMM:  // dims = {M, K, N}
      return gemm_split_workspace(M, F_or_N, H, dtype, EPI_BIAS);
    case TE_OP_LAYERNORM_DENSE_BWD:
      return dense_bwd_layout(nullptr, M, H, F_or_N, dtype, quantized != 0, kernel_dtype).bytes;
    default: return 0;
  }
}

te_status te_norm_fwd(const void* x, te_dtype x_dtype, int64_t M, int64_t H, const void* gamma,
                      const void* beta, te_norm_type norm_type, int zero_centered_gamma,
                      float epsilon, const te_quantizer* q, void* out, te_dtype out_dtype,
                      float* mu, float* rsigma, void* stream) {
  if (M < 0 || H <= 0 || !is_act_dtype(x_dtype) || out_dtype < TE_F32 || out_dtype > TE_E4M3 ||
      (norm_type != TE_LAYERNORM && norm_type != TE_RMSNORM))
    return TE_ERR_INVALID_ARG;
  if (M > 0 && (!x || !gamma || !out)) return TE_ERR_INVALID_ARG;
  if (out_dtype == TE_E4M3 && !enabled(q)) return TE_ERR_INVALID_ARG;
  if (!quantizer_ok(q)) return TE_ERR_INVALID_ARG;
  if (H % 8 || H * int64_t(esize(x_dtype)) > 16384) return TE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(gamma) || !opt_aligned16(beta) || !aligned16(out) ||
      !aligned4(mu) || !aligned4(rsigma))
    return TE_ERR_UNSUPPORTED;
  return norm_into(x, x_dtype, M, H, gamma, beta, norm_type, zero_centered_gamma, epsilon, q,
                   out, out_dtype, mu, rsigma, as_stream(stream));
}

te_status te_act_lu(const void* x, te_dtype x_dtype, int64_t M, int64_t N_in, te_act_type act,
                    const te_quantizer* q, void* out, te_dtype out_dtype, void* stream) {
  if (M < 0 || N_in <= 0 || !is_act_dtype(x_dtype) || !valid_act(act) ||
      out_dtype < TE_F32 || out_dtype > TE_E4M3)
    return TE_ERR_INVALID_ARG;
  if (M > 0 && (!x || !out)) return TE_ERR_INVALID_ARG;
  if (out_dtype == TE_E4M3 && !enabled(q)) return TE_ERR_INVALID_ARG;
  if (!quantizer_ok(q)) return TE_ERR_INVALID_ARG;
  const int64_t n_out = is_gated(act) ? N_in / 2 : N_in;
  if ((is_gated(act) && N_in % 2) || n_out % 8) return TE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(out)) return TE_ERR_UNSUPPORTED;
  if (M == 0) return TE_OK;
  const int fake = enabled(q) && out_dtype != TE_E4M3;
  return run_cast(q, out_dtype, fake, as_stream(stream), [&](const CastSpec& c) {
    ActArgs a;
    a.x = x;
    a.x_dtype = x_dtype;
    a.M = M;
    a.N_in = N_in;
    a.act = act;
    a.out = out;
    a.cast = c;
    return launch_act_lu(a, as_stream(stream));
  });
}

te_status te_dact_dbias_quantize(const void* dy, const void* x_preact, te_dtype dtype, int64_t M,
                                 int64_t N_in, te_act_type act, const te_quantizer* q, void* dx,
                                 te_dtype dx_dtype, float* dbias, void* workspace,
                                 size_t ws_bytes, void* stream) {
  if (M < 0 || N_in <= 0 || !is_act_dtype(dtype) || !valid_act(act) || dx_dtype < TE_F32 ||
      dx_dtype > TE_E4M3)
    return TE_ERR_INVALID_ARG;
  if (M > 0 && (!dy || (act != TE_IDENTITY && !x_preact) || !dx)) return TE_ERR_INVALID_ARG;
  if (dx_dtype == TE_E4M3 && !enabled(q)) return TE_ERR_INVALID_ARG;
  if (!quantizer_ok(q)) return TE_ERR_INVALID_ARG;
  const int64_t n_out = is_gated(act) ? N_in / 2 : N_in;
  if ((is_gated(act) && N_in % 2) || n_out % 8) return TE_ERR_UNSUPPORTED;
  if (!aligned16(dy) || !opt_aligned16(x_preact) || !aligned16(dx) || !aligned4(dbias))
    return TE_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  if (dbias && M == 0)
    return cudaMemsetAsync(dbias, 0, size_t(N_in) * 4, s) == cudaSuccess ? TE_OK : TE_ERR_CUDA;
  if (M == 0) return TE_OK;
  if (dbias && (!workspace || ws_bytes < dact_dbias_workspace(M, N_in))) return TE_ERR_WORKSPACE;
  if (dbias && !aligned16(workspace)) return TE_ERR_UNSUPPORTED;
  // Current scaling: dbias is reduced in the amax pass, the cast pass only stores dx.
  const bool two_pass = enabled(q) && q->mode == TE_SCALING_CURRENT;
  return run_cast(dx_dtype == TE_E4M3 ? q : nullptr, dx_dtype, 0, s, [&](const CastSpec& c) {
    DactArgs a;
    a.dy = dy;
    a.x = x_preact;
    a.dtype = dtype;
    a.M = M;
    a.N_in = N_in;
    a.act = act;
    a.dx = dx;
    const bool reduce_here = two_pass ? (c.store == 0) : true;
    a.dbias = reduce_here ? dbias : nullptr;
    a.partials = static_cast<float*>(workspace);
    a.cast = c;
    return launch_dact_dbias(a, s);
  });
}

te_status te_update_scales(const te_quantizer* qs, int n, void* stream) {
  if (n < 0 || n > kMaxScaleUpdates || (n > 0 && !qs)) return TE_ERR_INVALID_ARG;
  ScaleUpdateArgs a;
  for (int i = 0; i < n; ++i) {
    if (!enabled(&qs[i])) continue;  // a disabled quantizer has nothing to update
    if (!qs[i].amax || !aligned4(qs[i].amax) || !aligned4(qs[i].scale) ||
        !aligned4(qs[i].scale_inv))
      return TE_ERR_INVALID_ARG;
    a.amax[a.n] = qs[i].amax;
    a.scale[a.n] = qs[i].scale;
    a.scale_inv[a.n] = qs[i].scale_inv;
    ++a.n;
  }
  return launch_update_scales(a, as_stream(stream));
}

te_status te_quantize(const void* x, te_dtype x_dtype, int64_t M, int64_t N,
                      const te_quantizer* q, void* out, void* stream) {
  if (M < 0 || N <= 0 || !is_act_dtype(x_dtype) || !enabled(q)) return TE_ERR_INVALID_ARG;
  if (M > 0 && (!x || !out)) return TE_ERR_INVALID_ARG;
  if (!quantizer_ok(q)) return TE_ERR_INVALID_ARG;
  if (N % 8 || !aligned16(x) || !aligned16(out)) return TE_ERR_UNSUPPORTED;
  if (M == 0) return TE_OK;
  return quantize_into(x, x_dtype, M * N, q, out, as_stream(stream));
}

te_status te_gemm(const void* A, int a_trans, const void* B, int b_trans, te_dtype ab_dtype,
                  int64_t M, int64_t N, int64_t K, const float* a_scale_inv,
                  const float* b_scale_inv, const void* bias, te_dtype bias_dtype, void* D,
                  te_dtype d_dtype, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || N <= 0 || K <= 0 || ab_dtype < TE_F32 || ab_dtype > TE_E4M3 ||
      !is_act_dtype(d_dtype) || (bias && !is_act_dtype(bias_dtype)))
    return TE_ERR_INVALID_ARG;
  if (M > 0 && (!A || !B || !D)) return TE_ERR_INVALID_ARG;
  if (N % 16 || K % 16) return TE_ERR_UNSUPPORTED;
  if (a_trans && M % 16) return TE_ERR_UNSUPPORTED;  // M is then a row length
  // fp32 operands run as tf32, which the tensor cores take K-major only.
  if (ab_dtype == TE_F32 && (a_trans || !b_trans)) return TE_ERR_UNSUPPORTED;
  if (!aligned16(A) || !aligned16(B) || !aligned16(D) || !opt_aligned16(bias) ||
      !aligned4(a_scale_inv) || !aligned4(b_scale_inv) || !aligned16(workspace))
    return TE_ERR_UNSUPPORTED;
  if (M == 0) return TE_OK;
  GemmArgs g;
  g.split_ws = workspace;
  g.split_ws_bytes = workspace ? ws_bytes : 0;
  g.A = A;
  g.B = B;
  g.ab_dtype = ab_dtype;
  g.a_kmajor = a_trans ? 0 : 1;
  g.b_kmajor = b_trans ? 1 : 0;
  g.M = M;
  g.N = N;
  g.K = K;
  g.a_scale_inv = a_scale_inv;
  g.b_scale_inv = b_scale_inv;
  g.epilogue = EPI_BIAS;
  g.bias = bias;
  g.bias_dtype = bias_dtype;
  g.D = D;
  g.cast.out_dtype = d_dtype;
  return launch_gemm(g, as_stream(stream));
}

te_status te_layernorm_dense_fwd(const void* x, const void* kernel, te_dtype kernel_dtype,
                                 const void* gamma, const void* beta, const void* bias,
                                 te_norm_type norm_type, int zero_centered_gamma, float epsilon,
                                 const te_quantizer_set* qset, int64_t M, int64_t H, int64_t N,
                                 te_dtype dtype, void* out, void* saved_ln_out, float* mu,
                                 float* rsigma, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || H <= 0 || N <= 0 || !is_act_dtype(dtype) ||
      (norm_type != TE_LAYERNORM && norm_type != TE_RMSNORM))
    return TE_ERR_INVALID_ARG;
  const bool quant = qset != nullptr;
  if (quant) {
    if (!enabled(&qset->x) || !quantizer_ok(&qset->x) || !quantizer_ok(&qset->kernel1))
      return TE_ERR_INVALID_ARG;
    if (kernel_dtype == TE_E4M3 ? qset->kernel1.scale_inv == nullptr
                                : (kernel_dtype != dtype || !enabled(&qset->kernel1)))
      return TE_ERR_INVALID_ARG;
  } else if (kernel_dtype != dtype) {
    return TE_ERR_INVALID_ARG;
  }
  if (M > 0 && (!x || !kernel || !gamma || !out)) return TE_ERR_INVALID_ARG;
  if (H % 16 || N % 16 || H * int64_t(esize(dtype)) > 16384) return TE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(kernel) || !aligned16(gamma) || !opt_aligned16(beta) ||
      !opt_aligned16(bias) || !aligned16(out) || !opt_aligned16(saved_ln_out) ||
      !aligned16(workspace) || !aligned4(mu) || !aligned4(rsigma))
    return TE_ERR_UNSUPPORTED;
  if (M == 0) return TE_OK;
  FwdLayout L = dense_layout(workspace, M, H, N, dtype, quant, kernel_dtype, saved_ln_out != nullptr);
  if (L.split.required > 0 && (!workspace || ws_bytes < L.split.required)) return TE_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  void* ln = saved_ln_out ? saved_ln_out : L.ln;
  const int ln_dtype = quant ? TE_E4M3 : dtype;
  te_status st = norm_into(x, dtype, M, H, gamma, beta, norm_type, zero_centered_gamma, epsilon,
                           quant ? &qset->x : nullptr, ln, ln_dtype, mu, rsigma, s);
  if (st != TE_OK) return st;
  const void* kop = kernel;
  int b_kmajor = 0;
  if (quant && kernel_dtype != TE_E4M3) {
    st = quantize_into(kernel, dtype, H * N, &qset->kernel1, L.kq1, s);
    if (st != TE_OK) return st;
    kop = L.kq1;
  } else if (!quant && dtype == TE_F32) {
    st = launch_transpose_f32(static_cast<const float*>(kernel), H, N, static_cast<float*>(L.kt1), s);
    if (st != TE_OK) return st;
    kop = L.kt1;
    b_kmajor = 1;
  }
  GemmArgs g;
  g.A = ln;
  g.B = kop;
  g.ab_dtype = quant ? TE_E4M3 : dtype;
  g.a_kmajor = 1;
  g.b_kmajor = b_kmajor;
  g.M = M;
  g.N = N;
  g.K = H;
  g.a_scale_inv = quant ? qset->x.scale_inv : nullptr;
  g.b_scale_inv = quant ? qset->kernel1.scale_inv : nullptr;
  g.epilogue = EPI_BIAS;
  g.bias = bias;
  g.bias_dtype = dtype;
  g.D = out;
  g.cast.out_dtype = dtype;
  give_split(g, L.split, workspace, ws_bytes);
  return launch_gemm(g, s);
}

te_status te_layernorm_mlp_fwd(const void* x, const void* gamma, const void* beta,
                               const void* kernel1, const void* kernel2, te_dtype kernel_dtype,
                               const void* bias1, const void* bias2, te_norm_type norm_type,
                               int zero_centered_gamma, float epsilon, te_act_type act,
                               const te_quantizer_set* qset, int64_t M, int64_t H, int64_t F,
                               te_dtype dtype, void* out, void* saved_h, void* saved_act,
                               void* saved_ln_out, float* mu, float* rsigma, void* workspace,
                               size_t ws_bytes, void* stream) {
  if (M < 0 || H <= 0 || F <= 0 || !is_act_dtype(dtype) || act == TE_IDENTITY ||
      !valid_act(act) || (norm_type != TE_LAYERNORM && norm_type != TE_RMSNORM))
    return TE_ERR_INVALID_ARG;
  const bool quant = qset != nullptr;
  if (quant) {
    if (!enabled(&qset->x) || !enabled(&qset->act) || !quantizer_ok(&qset->x) ||
        !quantizer_ok(&qset->act) || !quantizer_ok(&qset->kernel1) || !quantizer_ok(&qset->kernel2))
      return TE_ERR_INVALID_ARG;
    if (kernel_dtype == TE_E4M3
            ? (!qset->kernel1.scale_inv || !qset->kernel2.scale_inv)
            : (kernel_dtype != dtype || !enabled(&qset->kernel1) || !enabled(&qset->kernel2)))
      return TE_ERR_INVALID_ARG;
  } else if (kernel_dtype != dtype) {
    return TE_ERR_INVALID_ARG;
  }
  if (M > 0 && (!x || !gamma || !kernel1 || !kernel2 || !out)) return TE_ERR_INVALID_ARG;
  if (H % 16 || F % 16 || H * int64_t(esize(dtype)) > 16384) return TE_ERR_UNSUPPORTED;
  if (!aligned16(x) || !aligned16(gamma) || !opt_aligned16(beta) || !aligned16(kernel1) ||
      !aligned16(kernel2) || !opt_aligned16(bias1) || !opt_aligned16(bias2) || !aligned16(out) ||
      !opt_aligned16(saved_h) || !opt_aligned16(saved_act) || !opt_aligned16(saved_ln_out) ||
      !aligned16(workspace) || !aligned4(mu) || !aligned4(rsigma))
    return TE_ERR_UNSUPPORTED;
  if (M == 0) return TE_OK;
  const bool gated = is_gated(act);
  const int64_t F1 = gated ? 2 * F : F;
  FwdLayout L = mlp_layout(workspace, M, H, F, dtype, quant, kernel_dtype, act,
                           saved_ln_out != nullptr);
  if (!workspace || ws_bytes < L.split.required) return TE_ERR_WORKSPACE;
  cudaStream_t s = as_stream(stream);
  void* ln = saved_ln_out ? saved_ln_out : L.ln;
  void* a2 = saved_act ? saved_act : L.a2;  // GEMM2's A operand
  // The activation's amax (GEMM1's epilogue accumulates into it) is zeroed before the norm rather
  // than between the norm and GEMM1, where the memset would keep GEMM1 from launching as the
  // norm's programmatic dependent; unless it shares storage with an amax written before GEMM1.
  const bool act_zero_first =
      quant && qset->act.amax && qset->act.amax != qset->x.amax &&
      (kernel_dtype == TE_E4M3 ||
       (qset->act.amax != qset->kernel1.amax && qset->act.amax != qset->kernel2.amax));
  te_status st = act_zero_first ? zero_scalar(qset->act.amax, s) : TE_OK;
  if (st != TE_OK) return st;
  // (1) normalization, written once in GEMM1's operand dtype
  st = norm_into(x, dtype, M, H, gamma, beta, norm_type, zero_centered_gamma, epsilon,
                 quant ? &qset->x : nullptr, ln, quant ? TE_E4M3 : dtype, mu, rsigma, s);
  if (st != TE_OK) return st;
  const void* w1 = kernel1;
  const void* w2 = kernel2;
  int b_kmajor = 0;
  if (quant && kernel_dtype != TE_E4M3) {
    st = quantize_into(kernel1, dtype, H * F1, &qset->kernel1, L.kq1, s);
    if (st != TE_OK) return st;
    st = quantize_into(kernel2, dtype, F * H, &qset->kernel2, L.kq2, s);
    if (st != TE_OK) return st;
    w1 = L.kq1;
    w2 = L.kq2;
  } else if (!quant && dtype == TE_F32) {
    st = launch_transpose_f32(static_cast<const float*>(kernel1), H, F1, static_cast<float*>(L.kt1), s);
    if (st != TE_OK) return st;
    st = launch_transpose_f32(static_cast<const float*>(kernel2), F, H, static_cast<float*>(L.kt2), s);
    if (st != TE_OK) return st;
    w1 = L.kt1;
    w2 = L.kt2;
    b_kmajor = 1;
  }
  // (2)+(3) GEMM1 + bias1 -> round -> activation [-> amax, E4M3], one kernel
  GemmArgs g1;
  g1.A = ln;
  g1.B = w1;
  g1.ab_dtype = quant ? TE_E4M3 : dtype;
  g1.a_kmajor = 1;
  g1.b_kmajor = b_kmajor;
  g1.M = M;
  g1.N = F1;
  g1.K = H;
  g1.a_scale_inv = quant ? qset->x.scale_inv : nullptr;
  g1.b_scale_inv = quant ? qset->kernel1.scale_inv : nullptr;
  g1.epilogue = gated ? EPI_BIAS_GATED : EPI_BIAS_ACT;
  g1.act = act;
  g1.bias = bias1;
  g1.bias_dtype = dtype;
  g1.h_dtype = dtype;
  g1.saved_h = saved_h;
  const bool act_current = quant && qset->act.mode == TE_SCALING_CURRENT;
  if (quant) {
    if (!act_zero_first) {
      st = zero_scalar(qset->act.amax, s);
      if (st != TE_OK) return st;
    }
    g1.cast.amax_out = qset->act.amax;
    if (act_current) {
      g1.D = L.a2_hi;
      g1.cast.out_dtype = TE_F32;
    } else {
      g1.D = a2;
      g1.cast.out_dtype = TE_E4M3;
      g1.cast.scale = qset->act.scale;
      g1.cast.scale_inv_out = qset->act.scale_inv;
    }
  } else {
    g1.D = a2;
    g1.cast.out_dtype = dtype;
  }
  give_split(g1, L.split, workspace, ws_bytes);
  st = launch_gemm(g1, s);
  if (st != TE_OK) return st;
  if (act_current) {
    // The amax is already known from GEMM1's epilogue: one cast pass.
    QuantizeArgs qa;
    qa.x = L.a2_hi;
    qa.x_dtype = TE_F32;
    qa.n = M * F;
    qa.out = a2;
    qa.cast.out_dtype = TE_E4M3;
    qa.cast.amax_in = qset->act.amax;
    qa.cast.scale_out = qset->act.scale;
    qa.cast.scale_inv_out = qset->act.scale_inv;
    st = launch_quantize(qa, s);
    if (st != TE_OK) return st;
  }
  // (4) GEMM2 + bias2
  GemmArgs g2;
  g2.A = a2;
  g2.B = w2;
  g2.ab_dtype = quant ? TE_E4M3 : dtype;
  g2.a_kmajor = 1;
  g2.b_kmajor = b_kmajor;
  g2.M = M;
  g2.N = H;
  g2.K = F;
  g2.a_scale_inv = quant ? qset->act.scale_inv : nullptr;
  g2.b_scale_inv = quant ? qset->kernel2.scale_inv : nullptr;
  g2.epilogue = EPI_BIAS;
  g2.bias = bias2;
  g2.bias_dtype = dtype;
  g2.D = out;
  g2.cast.out_dtype = dtype;
  give_split(g2, L.split, workspace, ws_bytes);
  return launch_gemm(g2, s);
}

te_status te_layernorm_mlp_bwd(const void* dy, const void* x, const void* gamma,
                               const void* kernel1, const void* kernel2, te_dtype kernel_dtype,
                               const void* saved_h, const void* saved_ln_out, const float* mu,
                               const float* rsigma, te_norm_type norm_type,
                               int zero_centered_gamma, te_act_type act,
                               const te_quantizer_set* qset, int64_t M, int64_t H, int64_t F,
                               te_dtype dtype, void* dx, float* dgamma, float* dbeta,
                               void* dkernel1, void* dkernel2, float* dbias1, float* dbias2,
                               void* saved_dh, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || H <= 0 || F <= 0 || dtype != TE_BF16 || act == TE_IDENTITY || !valid_act(act) ||
      (norm_type != TE_LAYERNORM && norm_type != TE_RMSNORM))
    return dtype == TE_F32 ? TE_ERR_UNSUPPORTED : TE_ERR_INVALID_ARG;
  const bool quant = qset != nullptr;
  if (quant) {
    if (!enabled(&qset->grad) || !quantizer_ok(&qset->grad) || !qset->x.scale_inv ||
        !quantizer_ok(&qset->kernel1))
      return TE_ERR_INVALID_ARG;
    if (kernel_dtype == TE_E4M3 ? !qset->kernel1.scale_inv
                                : (kernel_dtype != dtype || !enabled(&qset->kernel1)))
      return TE_ERR_INVALID_ARG;
  } else if (kernel_dtype != dtype) {
    return TE_ERR_INVALID_ARG;
  }
  if (!gamma || !dgamma || (M > 0 && (!dy || !x || !kernel1 || !kernel2 || !saved_h ||
                                      !saved_ln_out || !rsigma || !dx || !dkernel1 || !dkernel2)) ||
      (M > 0 && norm_type == TE_LAYERNORM && !mu))
    return TE_ERR_INVALID_ARG;
  if (H % 16 || F % 16 || H * int64_t(esize(dtype)) > 16384) return TE_ERR_UNSUPPORTED;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(kernel1) ||
      !aligned16(kernel2) || !aligned16(saved_h) || !aligned16(saved_ln_out) || !aligned16(dx) ||
      !aligned16(dkernel1) || !aligned16(dkernel2) || !aligned16(workspace) || !aligned4(mu) ||
      !aligned4(rsigma) || !aligned4(dgamma) || !aligned4(dbeta) || !aligned4(dbias1) ||
      !aligned4(dbias2) || !opt_aligned16(saved_dh))
    return TE_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  const bool gated = is_gated(act);
  const int64_t F1 = gated ? 2 * F : F;
  if (M == 0) {
    // no tokens: every gradient is zero
    const std::pair<void*, size_t> z[] = {{dgamma, size_t(H) * 4}, {dbeta, size_t(H) * 4},
                                          {dbias1, size_t(F1) * 4}, {dbias2, size_t(H) * 4},
                                          {dkernel1, size_t(H) * F1 * esize(dtype)},
                                          {dkernel2, size_t(F) * H * esize(dtype)}};
    for (const auto& e : z)
      if (e.first && cudaMemsetAsync(e.first, 0, e.second, s) != cudaSuccess) return TE_ERR_CUDA;
    return TE_OK;
  }
  BwdLayout L = bwd_layout(workspace, M, H, F, dtype, quant, kernel_dtype, act);
  if (!workspace || ws_bytes < L.split.required) return TE_ERR_WORKSPACE;
  float* partials = static_cast<float*>(L.partials);
  void* dh = saved_dh ? saved_dh : L.dh;  // the dgrad / wgrad GEMMs' operand
  te_status st;
  // dbias2 = column sums of dy
  if (dbias2) {
    DactArgs d;
    d.dy = dy;
    d.dtype = dtype;
    d.M = M;
    d.N_in = H;
    d.act = TE_IDENTITY;
    d.dx = nullptr;
    d.dbias = dbias2;
    d.partials = partials;
    st = launch_dact_dbias(d, s);
    if (st != TE_OK) return st;
  }
  // recompute the activation output (what GEMM2 consumed, in dtype)
  {
    ActArgs aa;
    aa.x = saved_h;
    aa.x_dtype = dtype;
    aa.M = M;
    aa.N_in = F1;
    aa.act = act;
    aa.out = L.a;
    aa.cast.out_dtype = dtype;
    st = launch_act_lu(aa, s);
    if (st != TE_OK) return st;
  }
  // dkernel2 = a^T dy   ([F, H], contraction over tokens)
  {
    GemmArgs g;
    g.A = L.a;
    g.B = dy;
    g.ab_dtype = dtype;
    g.a_kmajor = 0;
    g.b_kmajor = 0;
    g.M = F;
    g.N = H;
    g.K = M;
    g.D = dkernel2;
    g.cast.out_dtype = dtype;
    give_split(g, L.split, workspace, ws_bytes);
    st = launch_gemm(g, s);
    if (st != TE_OK) return st;
  }
  // da = dy kernel2^T   ([M, F], contraction over H)
  {
    GemmArgs g;
    g.A = dy;
    g.B = kernel2;
    g.ab_dtype = dtype;
    g.a_kmajor = 1;
    g.b_kmajor = 1;
    g.M = M;
    g.N = F;
    g.K = H;
    g.D = L.da;
    g.cast.out_dtype = dtype;
    give_split(g, L.split, workspace, ws_bytes);
    st = launch_gemm(g, s);
    if (st != TE_OK) return st;
  }
  // dH = da * act'(h), dbias1, quantized with the grad quantizer in FP8 mode
  st = run_cast(quant ? &qset->grad : nullptr, quant ? TE_E4M3 : dtype, 0, s,
                [&](const CastSpec& c) {
                  DactArgs d;
                  d.dy = L.da;
                  d.x = saved_h;
                  d.dtype = dtype;
                  d.M = M;
                  d.N_in = F1;
                  d.act = act;
                  d.dx = dh;
                  const bool two_pass = quant && qset->grad.mode == TE_SCALING_CURRENT;
                  d.dbias = (two_pass ? c.store == 0 : true) ? dbias1 : nullptr;
                  d.partials = partials;
                  d.cast = c;
                  return launch_dact_dbias(d, s);
                });
  if (st != TE_OK) return st;
  const void* w1 = kernel1;
  if (quant && kernel_dtype != TE_E4M3) {
    st = quantize_into(kernel1, dtype, H * F1, &qset->kernel1, L.kq1, s);
    if (st != TE_OK) return st;
    w1 = L.kq1;
  }
  // dln = dH kernel1^T   ([M, H], contraction over F')
  {
    GemmArgs g;
    g.A = dh;
    g.B = w1;
    g.ab_dtype = quant ? TE_E4M3 : dtype;
    g.a_kmajor = 1;
    g.b_kmajor = 1;
    g.M = M;
    g.N = H;
    g.K = F1;
    g.a_scale_inv = quant ? qset->grad.scale_inv : nullptr;
    g.b_scale_inv = quant ? qset->kernel1.scale_inv : nullptr;
    g.D = L.dln;
    g.cast.out_dtype = dtype;
    give_split(g, L.split, workspace, ws_bytes);
    st = launch_gemm(g, s);
    if (st != TE_OK) return st;
  }
  // dkernel1 = ln^T dH   ([H, F'], contraction over tokens)
  {
    GemmArgs g;
    g.A = saved_ln_out;
    g.B = dh;
    g.ab_dtype = quant ? TE_E4M3 : dtype;
    g.a_kmajor = 0;
    g.b_kmajor = 0;
    g.M = H;
    g.N = F1;
    g.K = M;
    g.a_scale_inv = quant ? qset->x.scale_inv : nullptr;
    g.b_scale_inv = quant ? qset->grad.scale_inv : nullptr;
    g.D = dkernel1;
    g.cast.out_dtype = dtype;
    give_split(g, L.split, workspace, ws_bytes);
    st = launch_gemm(g, s);
    if (st != TE_OK) return st;
  }
  // norm backward
  NormBwdArgs nb;
  nb.dz = L.dln;
  nb.x = x;
  nb.mu = mu;
  nb.rsigma = rsigma;
  nb.gamma = gamma;
  nb.dtype = dtype;
  nb.M = M;
  nb.H = H;
  nb.norm_type = norm_type;
  nb.zero_centered_gamma = zero_centered_gamma;
  nb.dx = dx;
  nb.dgamma = dgamma;
  nb.dbeta = norm_type == TE_LAYERNORM ? dbeta : nullptr;
  nb.partials = partials;
  // RMSNorm has no shift: the gradient of an (ignored) beta is zero
  if (norm_type == TE_RMSNORM && dbeta &&
      cudaMemsetAsync(dbeta, 0, size_t(H) * sizeof(float), s) != cudaSuccess)
    return TE_ERR_CUDA;
  return launch_norm_bwd(nb, s);
}

te_status te_layernorm_dense_bwd(const void* dy, const void* x, const void* gamma,
                                 const void* kernel, te_dtype kernel_dtype,
                                 const void* saved_ln_out, const float* mu, const float* rsigma,
                                 te_norm_type norm_type, int zero_centered_gamma,
                                 const te_quantizer_set* qset, int64_t M, int64_t H, int64_t N,
                                 te_dtype dtype, void* dx, float* dgamma, float* dbeta,
                                 void* dkernel, float* dbias, void* workspace, size_t ws_bytes,
                                 void* stream) {
  if (M < 0 || H <= 0 || N <= 0 || dtype != TE_BF16 ||
      (norm_type != TE_LAYERNORM && norm_type != TE_RMSNORM))
    return dtype == TE_F32 ? TE_ERR_UNSUPPORTED : TE_ERR_INVALID_ARG;
  const bool quant = qset != nullptr;
  if (quant) {
    if (!enabled(&qset->grad) || !quantizer_ok(&qset->grad) || !qset->x.scale_inv ||
        !quantizer_ok(&qset->kernel1))
      return TE_ERR_INVALID_ARG;
    if (kernel_dtype == TE_E4M3 ? !qset->kernel1.scale_inv
                                : (kernel_dtype != dtype || !enabled(&qset->kernel1)))
      return TE_ERR_INVALID_ARG;
  } else if (kernel_dtype != dtype) {
    return TE_ERR_INVALID_ARG;
  }
  if (!gamma || !dgamma || (M > 0 && (!dy || !x || !kernel || !saved_ln_out || !rsigma || !dx ||
                                      !dkernel)) ||
      (M > 0 && norm_type == TE_LAYERNORM && !mu))
    return TE_ERR_INVALID_ARG;
  if (H % 16 || N % 16 || H * int64_t(esize(dtype)) > 16384) return TE_ERR_UNSUPPORTED;
  if (!aligned16(dy) || !aligned16(x) || !aligned16(gamma) || !aligned16(kernel) ||
      !aligned16(saved_ln_out) || !aligned16(dx) || !aligned16(dkernel) || !aligned16(workspace) ||
      !aligned4(mu) || !aligned4(rsigma) || !aligned4(dgamma) || !aligned4(dbeta) ||
      !aligned4(dbias))
    return TE_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  if (M == 0) {
    // no tokens: every gradient is zero
    const std::pair<void*, size_t> z[] = {{dgamma, size_t(H) * 4}, {dbeta, size_t(H) * 4},
                                          {dbias, size_t(N) * 4},
                                          {dkernel, size_t(H) * N * esize(dtype)}};
    for (const auto& e : z)
      if (e.first && cudaMemsetAsync(e.first, 0, e.second, s) != cudaSuccess) return TE_ERR_CUDA;
    return TE_OK;
  }
  DenseBwdLayout L = dense_bwd_layout(workspace, M, H, N, dtype, quant, kernel_dtype);
  if (!workspace || ws_bytes < L.split.required) return TE_ERR_WORKSPACE;
  float* partials = static_cast<float*>(L.partials);
  te_status st;
  // dbias = column sums of dy; in FP8 mode the same pass casts dy with the grad quantizer
  if (quant) {
    st = run_cast(&qset->grad, TE_E4M3, 0, s, [&](const CastSpec& c) {
      DactArgs d;
      d.dy = dy;
      d.dtype = dtype;
      d.M = M;
      d.N_in = N;
      d.act = TE_IDENTITY;
      d.dx = L.dyq;
      const bool two_pass = qset->grad.mode == TE_SCALING_CURRENT;
      d.dbias = (two_pass ? c.store == 0 : true) ? dbias : nullptr;
      d.partials = partials;
      d.cast = c;
      return launch_dact_dbias(d, s);
    });
    if (st != TE_OK) return st;
  } else if (dbias) {
    DactArgs d;
    d.dy = dy;
    d.dtype = dtype;
    d.M = M;
    d.N_in = N;
    d.act = TE_IDENTITY;
    d.dx = nullptr;
    d.dbias = dbias;
    d.partials = partials;
    st = launch_dact_dbias(d, s);
    if (st != TE_OK) return st;
  }
  const void* gy = quant ? L.dyq : dy;
  const void* w = kernel;
  if (quant && kernel_dtype != TE_E4M3) {
    st = quantize_into(kernel, dtype, H * N, &qset->kernel1, L.kq, s);
    if (st != TE_OK) return st;
    w = L.kq;
  }
  // dln = dy kernel^T   ([M, H], contraction over N)
  {
    GemmArgs g;
    g.A = gy;
    g.B = w;
    g.ab_dtype = quant ? TE_E4M3 : dtype;
    g.a_kmajor = 1;
    g.b_kmajor = 1;
    g.M = M;
    g.N = H;
    g.K = N;
    g.a_scale_inv = quant ? qset->grad.scale_inv : nullptr;
    g.b_scale_inv = quant ? qset->kernel1.scale_inv : nullptr;
    g.D = L.dln;
    g.cast.out_dtype = dtype;
    give_split(g, L.split, workspace, ws_bytes);
    st = launch_gemm(g, s);
    if (st != TE_OK) return st;
  }
  // dkernel = ln^T dy   ([H, N], contraction over tokens)
  {
    GemmArgs g;
    g.A = saved_ln_out;
    g.B = gy;
    g.ab_dtype = quant ? TE_E4M3 : dtype;
    g.a_kmajor = 0;
    g.b_kmajor = 0;
    g.M = H;
    g.N = N;
    g.K = M;
    g.a_scale_inv = quant ? qset->x.scale_inv : nullptr;
    g.b_scale_inv = quant ? qset->grad.scale_inv : nullptr;
    g.D = dkernel;
    g.cast.out_dtype = dtype;
    give_split(g, L.split, workspace, ws_bytes);
    st = launch_gemm(g, s);
    if (st != TE_OK) return st;
  }
  NormBwdArgs nb;
  nb.dz = L.dln;
  nb.x = x;
  nb.mu = mu;
  nb.rsigma = rsigma;
  nb.gamma = gamma;
  nb.dtype = dtype;
  nb.M = M;
  nb.H = H;
  nb.norm_type = norm_type;
  nb.zero_centered_gamma = zero_centered_gamma;
  nb.dx = dx;
  nb.dgamma = dgamma;
  nb.dbeta = norm_type == TE_LAYERNORM ? dbeta : nullptr;
  nb.partials = partials;
  // RMSNorm has no shift: the gradient of an (ignored) beta is zero
  if (norm_type == TE_RMSNORM && dbeta &&
      cudaMemsetAsync(dbeta, 0, size_t(H) * sizeof(float), s) != cudaSuccess)
    return TE_ERR_CUDA;
  return launch_norm_bwd(nb, s);
}

te_status te_norm_bwd(const void* dz, const void* x, const float* mu, const float* rsigma,
                      const void* gamma, te_dtype dtype, int64_t M, int64_t H,
                      te_norm_type norm_type, int zero_centered_gamma, void* dx, float* dgamma,
                      float* dbeta, void* workspace, size_t ws_bytes, void* stream) {
  if (M < 0 || H <= 0 || !is_act_dtype(dtype) ||
      (norm_type != TE_LAYERNORM && norm_type != TE_RMSNORM))
    return TE_ERR_INVALID_ARG;
  if (!gamma || !dgamma || (M > 0 && (!dz || !x || !rsigma || !dx)) ||
      (M > 0 && norm_type == TE_LAYERNORM && !mu))
    return TE_ERR_INVALID_ARG;
  if (H % 8 || H * int64_t(esize(dtype)) > 16 * 4 * 256) return TE_ERR_UNSUPPORTED;
  if (!aligned16(dz) || !aligned16(x) || !aligned16(gamma) || !aligned16(dx) ||
      !aligned4(mu) || !aligned4(rsigma) || !aligned4(dgamma) || !aligned4(dbeta))
    return TE_ERR_UNSUPPORTED;
  cudaStream_t s = as_stream(stream);
  if (M == 0) {
    if (cudaMemsetAsync(dgamma, 0, size_t(H) * 4, s) != cudaSuccess) return TE_ERR_CUDA;
    if (dbeta && cudaMemsetAsync(dbeta, 0, size_t(H) * 4, s) != cudaSuccess) return TE_ERR_CUDA;
    return TE_OK;
  }
  if (!workspace || ws_bytes < norm_bwd_workspace(M, H)) return TE_ERR_WORKSPACE;
  if (!aligned16(workspace)) return TE_ERR_UNSUPPORTED;
  NormBwdArgs a;
  a.dz = dz;
  a.x = x;
  a.mu = mu;
  a.rsigma = rsigma;
  a.gamma = gamma;
  a.dtype = dtype;
  a.M = M;
  a.H = H;
  a.norm_type = norm_type;
  a.zero_centered_gamma = zero_centered_gamma;
  a.dx = dx;
  a.dgamma = dgamma;
  a.dbeta = norm_type == TE_LAYERNORM ? dbeta : nullptr;
  a.partials = static_cast<float*>(workspace);
  return launch_norm_bwd(a, s);
}

}  // extern "C"
