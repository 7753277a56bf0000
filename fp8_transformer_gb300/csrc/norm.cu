// Row normalization kernels (LayerNorm / RMSNorm forward and backward).
//
// Forward (TransformerEngine JAX "LayerNorm MLP" page, Description step (1); "LayerNorm Dense"
// page, Description): one warp per row, rows streamed into a per-warp double buffer in shared
// memory by the bulk-copy engine, fp32 statistics, and the normalized row written once,
// directly in the consumer GEMM's operand dtype (fp32, bf16 or E4M3) with 16-byte stores,
// together with the per-tensor amax.
//
// Backward (the norm's share of the backward pass, whose gradients cover every parameter): one CTA walks
// a strided set of rows; each row's dx needs two row sums, reduced across the CTA; dgamma and
// dbeta accumulate per thread in registers, are written as one partial row per CTA and summed
// in a fixed order by a second kernel, so the result does not depend on timing.
#include "cast.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace te {

namespace {

constexpr int kFwdMaxWarps = 8;
constexpr size_t kFwdSmemBudget = 200 * 1024;  // row buffers per CTA

// One warp per row, persistent over rows.  Each warp owns two row buffers in shared memory:
// while it normalizes row r from one buffer, the bulk-copy engine streams row r + stride into
// the other, so every warp keeps a whole row in flight with few registers.
template <typename T>
__global__ void __launch_bounds__(kFwdMaxWarps * 32) norm_fwd_kernel(NormFwdArgs a, int* status,
                                                                     uint32_t row_bytes) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem) + 2 * warp;
  uint8_t* bufs = smem + 256 + size_t(warp) * 2 * row_bytes;
  if (lane == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    mbar_init_fence();
  }
  __syncwarp();
  const CastState cs = cast_begin(a.cast);
  const int nvec = int(a.H / E);
  const float inv_h = 1.0f / float(a.H);
  const bool ln = a.norm_type == TE_LAYERNORM;
  const int64_t stride = int64_t(gridDim.x) * nwarps;
  const char* xg = static_cast<const char*>(a.x);
  int issued[2] = {0, 0}, waited[2] = {0, 0};  // lane 0's bookkeeping of its copies
  float amax = 0.0f;
  int64_t row = int64_t(blockIdx.x) * nwarps + warp;
  if (lane == 0 && row < a.M) {
    mbar_expect_tx(smem_u32(&bars[0]), row_bytes);
    bulk_load(smem_u32(bufs), xg + row * row_bytes, row_bytes, smem_u32(&bars[0]));
    issued[0]++;
  }
  for (int i = 0; row < a.M; ++i, row += stride) {
    const int st = i & 1;
    const uint32_t par = uint32_t(i >> 1) & 1u;
    const int64_t next = row + stride;
    if (lane == 0 && next < a.M) {
      // the other buffer was last read in the previous iteration (ordered by __syncwarp)
      fence_proxy_async_smem();
      mbar_expect_tx(smem_u32(&bars[st ^ 1]), row_bytes);
      bulk_load(smem_u32(bufs + (st ^ 1) * row_bytes), xg + next * row_bytes, row_bytes,
                smem_u32(&bars[st ^ 1]));
      issued[st ^ 1]++;
    }
    int ok = 1;
    if (lane == 0) {
      ok = wait_bounded(smem_u32(&bars[st]), par, nullptr, status, kWaitLimitNs, false) ? 1 : 0;
      waited[st] += ok;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok) break;
    while (!mbar_try_wait(smem_u32(&bars[st]), par)) {
    }
    __syncwarp();
    const uint4* xs = reinterpret_cast<const uint4*>(bufs + st * row_bytes);
    float mean = 0.0f, rs;
    if (ln) {
      float s1 = 0.0f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float xv[E];
        V::unpack(xs[v], xv);
#pragma unroll
        for (int e = 0; e < E; ++e) s1 += xv[e];
      }
      mean = warp_sum(s1) * inv_h;
      float s2 = 0.0f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float xv[E];
        V::unpack(xs[v], xv);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float d = xv[e] - mean;
          s2 += d * d;
        }
      }
      rs = 1.0f / sqrtf(warp_sum(s2) * inv_h + a.eps);
    } else {
      float s2 = 0.0f;
#pragma unroll 4
      for (int v = lane; v < nvec; v += 32) {
        float xv[E];
        V::unpack(xs[v], xv);
#pragma unroll
        for (int e = 0; e < E; ++e) s2 += xv[e] * xv[e];
      }
      rs = 1.0f / sqrtf(warp_sum(s2) * inv_h + a.eps);
    }
    if (lane == 0) {
      if (a.mu) a.mu[row] = mean;
      if (a.rsigma) a.rsigma[row] = rs;
    }
    if (cs.store || a.cast.amax_out) {
#pragma unroll 2
      for (int v = lane; v < nvec; v += 32) {
        float xv[E], g[E], b[E], y[E];
        V::unpack(xs[v], xv);
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
    }
    __syncwarp();
  }
  // Copies still in flight land before the CTA may exit (only after a timeout).
  if (lane == 0) {
    for (int s2 = 0; s2 < 2; ++s2)
      if (issued[s2] > waited[s2])
        wait_bounded(smem_u32(&bars[s2]), uint32_t(waited[s2]) & 1u, nullptr, status,
                     kDrainLimitNs, false);
  }
  amax = warp_max(amax);
  if (lane == 0 && a.cast.amax_out) atomic_max_nonneg(a.cast.amax_out, amax);
}

template <typename T>
te_status launch_fwd_t(const NormFwdArgs& a, cudaStream_t s) {
  const uint32_t row_bytes = uint32_t(a.H * sizeof(T));
  int warps = int(kFwdSmemBudget / (2 * size_t(row_bytes)));
  if (warps < 1) return TE_ERR_UNSUPPORTED;
  if (warps > kFwdMaxWarps) warps = kFwdMaxWarps;
  const size_t smem = 256 + size_t(warps) * 2 * row_bytes;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    if (cudaFuncSetAttribute(norm_fwd_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(256 + kFwdSmemBudget)) != cudaSuccess)
      return TE_ERR_CUDA;
    attr_set[dev & 63] = true;
  }
  int per_sm = int((227 * 1024) / smem);
  if (per_sm < 1) per_sm = 1;
  if (per_sm * warps > 64) per_sm = 64 / warps;
  const int64_t needed = ceil_div(a.M, warps);
  const int64_t cap = int64_t(num_sms()) * per_sm;
  const unsigned grid = unsigned(needed < cap ? needed : cap);
  norm_fwd_kernel<T><<<grid, warps * 32, smem, s>>>(a, device_status_ptr(), row_bytes);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
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
  if (a.x_dtype == TE_BF16) return launch_fwd_t<__nv_bfloat16>(a, s);
  if (a.x_dtype == TE_F32) return launch_fwd_t<float>(a, s);
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
