// Row normalization kernels (LayerNorm / RMSNorm forward and backward).
//
// Forward (TransformerEngine JAX "LayerNorm MLP" page, Description step (1); "LayerNorm Dense"
// page, Description): one warp per row, rows streamed into a per-warp double buffer in shared
// memory by the bulk-copy engine, fp32 statistics, and the normalized row written once,
// directly in the consumer GEMM's operand dtype (fp32, bf16 or E4M3) with 16-byte stores,
// together with the per-tensor amax.
//
// Backward (the norm's share of the backward pass, whose gradients cover every parameter): one
// CTA walks strided groups of four rows; each row's dx needs two row sums, reduced across the
// CTA for the whole group at one barrier; dgamma and dbeta accumulate per thread in registers,
// are written as one partial row per CTA and summed in a fixed order by a second kernel, so the
// result does not depend on timing.
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
        with_out(out_kind(cs), [&](auto tag) {
          store_out<decltype(tag)::value, E>(a.out, row * a.H + int64_t(v) * E, y, cs);
        });
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

// Rows of up to 8 KB: one warp per row with the row resident in registers as packed 16-byte
// vectors, persistent over rows, 2+ CTAs per SM so that many rows are in flight per SM.  The
// gain (gamma, or 1 + gamma) and beta are expanded to fp32 in shared memory once per CTA, and
// the arithmetic runs on packed fp32 pairs.  Statistics take one pass, shifted by the row's
// first element (mean = x0 + E[x - x0], var = E[(x - x0)^2] - E[x - x0]^2), which avoids the
// cancellation of the unshifted form.
template <typename T, int NV>
__global__ void __launch_bounds__(256, 2) norm_fwd_reg_kernel(NormFwdArgs a) {
  using V = Vec16<T>;
  using PR = Pairs<T>;
  constexpr int E = V::N;
  constexpr int P = PR::P;
  // gain (gamma, or 1 + gamma) and beta in fp32, laid out as float4 blocks so that the lanes of
  // a warp, which own consecutive 16-byte input vectors, read consecutive float4s:
  // element e of vector v sits in block (e / 4) * nvec + v, slot e % 4.
  extern __shared__ float4 params[];
  const int nvec = int(a.H / E);
  constexpr int Q = E / 4;
  float4* gain4 = params;
  float4* beta4 = params + Q * nvec;
  const bool ln = a.norm_type == TE_LAYERNORM;
  {
    const float shift = a.zero_centered_gamma ? 1.0f : 0.0f;
    const T* g = static_cast<const T*>(a.gamma);
    const T* b = static_cast<const T*>(a.beta);
    float* gf = reinterpret_cast<float*>(gain4);
    float* bf = reinterpret_cast<float*>(beta4);
    for (int64_t j = threadIdx.x; j < a.H; j += blockDim.x) {
      const int64_t v = j / E, e = j % E;
      const int64_t slot = ((e / 4) * nvec + v) * 4 + (e % 4);
      gf[slot] = float(g[j]) + shift;
      bf[slot] = (ln && b) ? float(b[j]) : 0.0f;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const CastState cs = cast_begin(a.cast);
  const float inv_h = 1.0f / float(a.H);
  const bool want_amax = a.cast.amax_out != nullptr;
  float amax = 0.0f;
  with_out(out_kind(cs), [&](auto tag) {
  constexpr int OUT = decltype(tag)::value;
  for (int64_t row = int64_t(blockIdx.x) * nwarps + warp; row < a.M;
       row += int64_t(gridDim.x) * nwarps) {
    const T* xr = static_cast<const T*>(a.x) + row * a.H;
    uint4 raw[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = lane + i * 32;
      raw[i] = v < nvec ? __ldg(reinterpret_cast<const uint4*>(xr) + v) : make_uint4(0u, 0u, 0u, 0u);
    }
    float x0 = 0.0f;
    if (ln) {
      f32x2 first[P];
      PR::get(raw[0], first);
      x0 = __shfl_sync(0xffffffffu, f2lo(first[0]), 0);
    }
    const f32x2 x02 = f2s(x0);
    f32x2 s1 = f2s(0.0f), s2 = f2s(0.0f);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      if (lane + i * 32 < nvec) {
        f32x2 xp[P];
        PR::get(raw[i], xp);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          const f32x2 d = sub2(xp[p], x02);
          s1 = add2(s1, d);
          s2 = fma2(d, d, s2);
        }
      }
    }
    const float m1 = warp_sum(f2lo(s1) + f2hi(s1)) * inv_h;
    const float m2 = warp_sum(f2lo(s2) + f2hi(s2)) * inv_h;
    const float mean = ln ? x0 + m1 : 0.0f;
    const float var = ln ? fmaxf(m2 - m1 * m1, 0.0f) : m2;
    const float rs = 1.0f / sqrtf(var + a.eps);
    if (lane == 0) {
      if (a.mu) a.mu[row] = mean;
      if (a.rsigma) a.rsigma[row] = rs;
    }
    if (OUT != OUT_NONE || want_amax) {
      const f32x2 mean2 = f2s(mean), rs2 = f2s(rs);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int v = lane + i * 32;
        if (v < nvec) {
          f32x2 xp[P], gp[P], bp[P];
          PR::get(raw[i], xp);
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            const float4 g4 = gain4[q * nvec + v];
            const float4 b4 = beta4[q * nvec + v];
            gp[2 * q] = f2(g4.x, g4.y);
            gp[2 * q + 1] = f2(g4.z, g4.w);
            bp[2 * q] = f2(b4.x, b4.y);
            bp[2 * q + 1] = f2(b4.z, b4.w);
          }
          float y[E];
#pragma unroll
          for (int p = 0; p < P; ++p) {
            const f32x2 yy = fma2(sub2(xp[p], mean2), mul2(gp[p], rs2), bp[p]);
            if (want_amax) amax = absmax2(amax, yy);
            y[2 * p] = f2lo(yy);
            y[2 * p + 1] = f2hi(yy);
          }
          store_out<OUT, E>(a.out, row * a.H + int64_t(v) * E, y, cs);
        }
      }
    }
  }
  });
  amax = warp_max(amax);
  if (lane == 0 && a.cast.amax_out) atomic_max_nonneg(a.cast.amax_out, amax);
}

template <typename T>
te_status launch_fwd_smem(const NormFwdArgs& a, cudaStream_t s);

template <typename T, int NV>
te_status launch_fwd_reg(const NormFwdArgs& a, cudaStream_t s) {
  const int warps = 8;
  const size_t smem = size_t(a.H) * 2 * sizeof(float);  // fp32 gain and beta
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm_fwd_reg_kernel<T, NV>,
                                                    warps * 32, smem) != cudaSuccess || per_sm < 1)
    per_sm = 1;
  const int64_t needed = ceil_div(a.M, warps);
  const int64_t cap = int64_t(num_sms()) * per_sm;
  const unsigned grid = unsigned(needed < cap ? needed : cap);
  norm_fwd_reg_kernel<T, NV><<<grid, warps * 32, smem, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T>
te_status launch_fwd_t(const NormFwdArgs& a, cudaStream_t s) {
  constexpr int E = Vec16<T>::N;
  const int64_t per_lane = ceil_div(a.H / E, 32);
  if (per_lane <= 1) return launch_fwd_reg<T, 1>(a, s);
  if (per_lane <= 2) return launch_fwd_reg<T, 2>(a, s);
  if (per_lane <= 4) return launch_fwd_reg<T, 4>(a, s);
  if (per_lane <= 8) return launch_fwd_reg<T, 8>(a, s);
  if (per_lane <= 16) return launch_fwd_reg<T, 16>(a, s);
  return launch_fwd_smem<T>(a, s);
}

// Longer rows: streamed through per-warp shared-memory double buffers (norm_fwd_kernel).
template <typename T>
te_status launch_fwd_smem(const NormFwdArgs& a, cudaStream_t s) {
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
constexpr int kBwdRows = 4;  // rows per CTA between two barriers, for rows of <= 4 KB

// Rows per barrier for NV vectors per thread (the first pass holds the group's x and dz in
// registers).
__host__ __device__ constexpr int bwd_rows(int nv) { return nv >= 4 ? 2 : 4; }

// One CTA per group of kBwdRows rows at a time (persistent over groups).  Each row's dx needs
// two row sums; the CTA reduces the sums of all its rows with one barrier.  dgamma / dbeta
// accumulate per thread in registers over every row the CTA visits.
template <typename T, int NV>
__global__ void __launch_bounds__(kBwdThreads, 2) norm_bwd_kernel(NormBwdArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  constexpr int R = bwd_rows(NV);
  __shared__ float red[2][kBwdWarps][R][2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nvec = int(a.H / E);
  const float inv_h = 1.0f / float(a.H);
  const bool ln = a.norm_type == TE_LAYERNORM;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  uint4 graw[NV];
  float accg[NV][E], accb[NV][E];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = tid + i * kBwdThreads;
    graw[i] = v < nvec ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.gamma)) + v) : zero;
#pragma unroll
    for (int e = 0; e < E; ++e) { accg[i][e] = 0.0f; accb[i][e] = 0.0f; }
  }
  const float gshift = a.zero_centered_gamma ? 1.0f : 0.0f;
  int parity = 0;
  for (int64_t r0 = int64_t(blockIdx.x) * R; r0 < a.M; r0 += int64_t(gridDim.x) * R, parity ^= 1) {
    uint4 rx[R][NV], rdz[R][NV];
    float mu[R], rs[R];
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int64_t row = r0 + j;
      const bool in = row < a.M;
      mu[j] = (in && ln) ? a.mu[row] : 0.0f;
      rs[j] = in ? a.rsigma[row] : 0.0f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int v = tid + i * kBwdThreads;
        const bool ok = in && v < nvec;
        rx[j][i] = ok ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + row * a.H) + v) : zero;
        rdz[j][i] = ok ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dz) + row * a.H) + v) : zero;
      }
    }
#pragma unroll
    for (int j = 0; j < R; ++j) {
      float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        float xv[E], dz[E], g[E];
        V::unpack(rx[j][i], xv);
        V::unpack(rdz[j][i], dz);
        V::unpack(graw[i], g);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float dyg = dz[e] * (g[e] + gshift);
          s1 += dyg;
          s2 += dyg * ((xv[e] - mu[j]) * rs[j]);
        }
      }
      s1 = warp_sum(s1);
      s2 = warp_sum(s2);
      if (lane == 0) {
        red[parity][warp][j][0] = s1;
        red[parity][warp][j][1] = s2;
      }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < R; ++j) {
      const int64_t row = r0 + j;
      if (row >= a.M) break;
      float s1 = 0.0f, s2 = 0.0f;
#pragma unroll
      for (int w = 0; w < kBwdWarps; ++w) {
        s1 += red[parity][w][j][0];
        s2 += red[parity][w][j][1];
      }
      const float m1 = ln ? s1 * inv_h : 0.0f;
      const float m2 = s2 * inv_h;
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int v = tid + i * kBwdThreads;
        if (v < nvec) {
          // x and dz come again from cache (L1/L2): keeping the group's rows in registers
          // across the barrier would spill.
          float xv[E], dz[E], g[E], dx[E];
          V::unpack(ldg16_ordered(static_cast<const T*>(a.x) + row * a.H + int64_t(v) * E), xv);
          V::unpack(ldg16_ordered(static_cast<const T*>(a.dz) + row * a.H + int64_t(v) * E), dz);
          V::unpack(graw[i], g);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float xh = (xv[e] - mu[j]) * rs[j];
            dx[e] = rs[j] * (dz[e] * (g[e] + gshift) - m1 - xh * m2);
            accg[i][e] += dz[e] * xh;
            accb[i][e] += dz[e];
          }
          store_out<(E == 8 ? OUT_BF16 : OUT_F32), E>(a.dx, row * a.H + int64_t(v) * E, dx,
                                                      CastState{});
        }
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

int bwd_chunks(int64_t M) {
  // enough row groups for the smallest group size (one row), capped at the resident CTAs
  const int64_t groups = M;
  const int64_t resident = int64_t(num_sms()) * 2;
  return int(groups < resident ? groups : resident);
}

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
