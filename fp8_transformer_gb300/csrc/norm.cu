// Row normalization kernels (LayerNorm / RMSNorm forward and backward).
//
// Forward (TransformerEngine JAX "LayerNorm MLP" page, Description step (1); "LayerNorm Dense"
// page, Description): one warp per row, the row held in registers as 16-byte vectors, fp32
// statistics, and the normalized row written once, directly in the consumer GEMM's operand
// dtype (fp32, bf16 or E4M3) together with the per-tensor amax.
//
// Backward (the norm's share of the backward pass, whose gradients cover every parameter): one CTA walks
// a strided set of rows; each row's dx needs two row sums, reduced across the CTA; dgamma and
// dbeta accumulate per thread in registers, are written as one partial row per CTA and summed
// in a fixed order by a second kernel, so the result does not depend on timing.
#include "cast.cuh"
#include "common.cuh"
#include "kernels.h"

namespace te {

namespace {

constexpr int kFwdWarps = 8;

template <typename T, int NV>
__global__ void __launch_bounds__(kFwdWarps * 32) norm_fwd_kernel(NormFwdArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * kFwdWarps + warp;
  const CastState cs = cast_begin(a.cast);
  float amax = 0.0f;
  if (row < a.M) {
    const int nvec = int(a.H / E);
    const T* xr = static_cast<const T*>(a.x) + row * a.H;
    const uint4* xr16 = reinterpret_cast<const uint4*>(xr);
    // The row stays in registers as raw 16-byte vectors and is unpacked on each pass.
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = lane + i * 32;
      raw[i] = v < nvec ? __ldg(xr16 + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    const float inv_h = 1.0f / float(a.H);
    float mean = 0.0f, rs;
    if (a.norm_type == TE_LAYERNORM) {
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        float xv[E];
        V::unpack(raw[i], xv);
#pragma unroll
        for (int e = 0; e < E; ++e) s += xv[e];
      }
      mean = warp_sum(s) * inv_h;
      float ss = 0.0f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        if (lane + i * 32 < nvec) {
          float xv[E];
          V::unpack(raw[i], xv);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float d = xv[e] - mean;
            ss += d * d;
          }
        }
      }
      rs = 1.0f / sqrtf(warp_sum(ss) * inv_h + a.eps);
    } else {
      float ss = 0.0f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        float xv[E];
        V::unpack(raw[i], xv);
#pragma unroll
        for (int e = 0; e < E; ++e) ss += xv[e] * xv[e];
      }
      rs = 1.0f / sqrtf(warp_sum(ss) * inv_h + a.eps);
    }
    if (lane == 0) {
      if (a.mu) a.mu[row] = mean;
      if (a.rsigma) a.rsigma[row] = rs;
    }
    const bool ln = a.norm_type == TE_LAYERNORM;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = lane + i * 32;
      if (v < nvec) {
        float xv[E], g[E], b[E], y[E];
        // Re-read from cache rather than keeping the packed row alive through this pass.
        V::load(xr, int64_t(v) * E, xv);
        V::load(a.gamma, int64_t(v) * E, g);
        if (ln && a.beta) {
          V::load(a.beta, int64_t(v) * E, b);
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) b[e] = 0.0f;
        }
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float gain = a.zero_centered_gamma ? 1.0f + g[e] : g[e];
          y[e] = (xv[e] - mean) * rs * gain + b[e];
          amax = fmaxf(amax, fabsf(y[e]));
        }
        if (cs.store) cast_store<E>(a.out, row * a.H + int64_t(v) * E, y, cs);
      }
      // Keeps the next vector's gamma/beta loads from being hoisted above this store, which
      // would hold every vector's parameters in registers at once.
      asm volatile("" ::: "memory");
    }
  }
  block_amax_commit(amax, a.cast.amax_out);
}

template <typename T, int NV>
te_status launch_fwd_t(const NormFwdArgs& a, cudaStream_t s) {
  const unsigned grid = unsigned(ceil_div(a.M, kFwdWarps));
  norm_fwd_kernel<T, NV><<<grid, kFwdWarps * 32, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T>
te_status launch_fwd_dispatch(const NormFwdArgs& a, cudaStream_t s) {
  constexpr int E = Vec16<T>::N;
  const int64_t per_lane = ceil_div(a.H / E, 32);
  if (per_lane <= 1) return launch_fwd_t<T, 1>(a, s);
  if (per_lane <= 2) return launch_fwd_t<T, 2>(a, s);
  if (per_lane <= 4) return launch_fwd_t<T, 4>(a, s);
  if (per_lane <= 8) return launch_fwd_t<T, 8>(a, s);
  if (per_lane <= 16) return launch_fwd_t<T, 16>(a, s);
  if (per_lane <= 32) return launch_fwd_t<T, 32>(a, s);
  return TE_ERR_UNSUPPORTED;
}

// ----------------------------------------------------------------------- backward --------

constexpr int kBwdThreads = 256;
constexpr int kBwdWarps = kBwdThreads / 32;

template <typename T, int NV>
__global__ void __launch_bounds__(kBwdThreads) norm_bwd_kernel(NormBwdArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  __shared__ float red[2][kBwdWarps][2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = int(a.H / E);
  const float inv_h = 1.0f / float(a.H);
  const bool ln = a.norm_type == TE_LAYERNORM;
  float g[NV][E], accg[NV][E], accb[NV][E];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = tid + i * kBwdThreads;
#pragma unroll
    for (int e = 0; e < E; ++e) { accg[i][e] = 0.0f; accb[i][e] = 0.0f; g[i][e] = 0.0f; }
    if (v < nvec) {
      V::load(a.gamma, int64_t(v) * E, g[i]);
      if (a.zero_centered_gamma)
#pragma unroll
        for (int e = 0; e < E; ++e) g[i][e] += 1.0f;
    }
  }
  int parity = 0;
  for (int64_t row = blockIdx.x; row < a.M; row += gridDim.x, parity ^= 1) {
    const float mu = ln ? a.mu[row] : 0.0f;
    const float rs = a.rsigma[row];
    float xh[NV][E], dz[NV][E];
    float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = tid + i * kBwdThreads;
      if (v < nvec) {
        V::load(a.x, row * a.H + int64_t(v) * E, xh[i]);
        V::load(a.dz, row * a.H + int64_t(v) * E, dz[i]);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          xh[i][e] = (xh[i][e] - mu) * rs;
          const float dyg = dz[i][e] * g[i][e];
          s1 += dyg;
          s2 += dyg * xh[i][e];
        }
      }
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    if (lane == 0) { red[parity][warp][0] = s1; red[parity][warp][1] = s2; }
    __syncthreads();
    s1 = 0.0f; s2 = 0.0f;
#pragma unroll
    for (int w = 0; w < kBwdWarps; ++w) { s1 += red[parity][w][0]; s2 += red[parity][w][1]; }
    const float m1 = ln ? s1 * inv_h : 0.0f;
    const float m2 = s2 * inv_h;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = tid + i * kBwdThreads;
      if (v < nvec) {
        float dx[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          dx[e] = rs * (dz[i][e] * g[i][e] - m1 - xh[i][e] * m2);
          accg[i][e] += dz[i][e] * xh[i][e];
          accb[i][e] += dz[i][e];
        }
        CastState cs;
        cs.out_dtype = a.dtype;
        cast_store<E>(a.dx, row * a.H + int64_t(v) * E, dx, cs);
      }
    }
  }
  float* pg = a.partials + int64_t(blockIdx.x) * 2 * a.H;
  float* pb = pg + a.H;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = tid + i * kBwdThreads;
    if (v < nvec) {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        pg[int64_t(v) * E + e] = accg[i][e];
        pb[int64_t(v) * E + e] = accb[i][e];
      }
    }
  }
}

// dgamma[j] = sum_c partials[c][0][j], dbeta[j] = sum_c partials[c][1][j], in chunk order.
__global__ void norm_bwd_reduce_kernel(const float* partials, int chunks, int64_t H,
                                       float* dgamma, float* dbeta) {
  const int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= H) return;
  float sg = 0.0f, sb = 0.0f;
  for (int c = 0; c < chunks; ++c) {
    sg += partials[int64_t(c) * 2 * H + j];
    sb += partials[int64_t(c) * 2 * H + H + j];
  }
  dgamma[j] = sg;
  if (dbeta) dbeta[j] = sb;
}

int bwd_chunks(int64_t M) { return int(M < int64_t(num_sms()) * 4 ? M : int64_t(num_sms()) * 4); }

template <typename T, int NV>
te_status launch_bwd_t(const NormBwdArgs& a, cudaStream_t s) {
  const int chunks = bwd_chunks(a.M);
  norm_bwd_kernel<T, NV><<<chunks, kBwdThreads, 0, s>>>(a);
  norm_bwd_reduce_kernel<<<unsigned(ceil_div(a.H, 256)), 256, 0, s>>>(a.partials, chunks, a.H,
                                                                       a.dgamma, a.dbeta);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T>
te_status launch_bwd_dispatch(const NormBwdArgs& a, cudaStream_t s) {
  constexpr int E = Vec16<T>::N;
  const int64_t per_thread = ceil_div(a.H / E, kBwdThreads);
  if (per_thread <= 1) return launch_bwd_t<T, 1>(a, s);
  if (per_thread <= 2) return launch_bwd_t<T, 2>(a, s);
  if (per_thread <= 4) return launch_bwd_t<T, 4>(a, s);
  return TE_ERR_UNSUPPORTED;
}

}  // namespace

te_status launch_norm_fwd(const NormFwdArgs& a, cudaStream_t s) {
  if (a.M == 0) return TE_OK;
  ProfileScope prof(TE_KERNEL_NORM_FWD, s);
  if (a.x_dtype == TE_BF16) return launch_fwd_dispatch<__nv_bfloat16>(a, s);
  if (a.x_dtype == TE_F32) return launch_fwd_dispatch<float>(a, s);
  return TE_ERR_UNSUPPORTED;
}

size_t norm_bwd_workspace(int64_t M, int64_t H) {
  return size_t(bwd_chunks(M > 0 ? M : 1)) * 2 * size_t(H) * sizeof(float);
}

te_status launch_norm_bwd(const NormBwdArgs& a, cudaStream_t s) {
  if (a.M == 0) return TE_OK;
  ProfileScope prof(TE_KERNEL_NORM_BWD, s);
  if (a.dtype == TE_BF16) return launch_bwd_dispatch<__nv_bfloat16>(a, s);
  if (a.dtype == TE_F32) return launch_bwd_dispatch<float>(a, s);
  return TE_ERR_UNSUPPORTED;
}

}  // namespace te
