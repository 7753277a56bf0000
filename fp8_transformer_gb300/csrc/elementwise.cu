// Bandwidth-bound kernels of the block that need no staging: the per-tensor quantize and the
// fp32 transpose of the tf32 path.  (The activation and the backward's activation gradient +
// bias reduction + quantize stream through TMA in stream.cu.)
//
// * quantize (TransformerEngine JAX "LayerNorm Dense" page, Description: the normalized output
//   and the kernel are quantized before the GEMM): 16-byte vectors, grid-stride, amax by one
//   integer atomic per block.
#include "cast.cuh"
#include "common.cuh"
#include "kernels.h"

namespace te {

namespace {

constexpr int kEwThreads = 256;

unsigned ew_grid(int64_t vectors) {
  const int64_t per_wave = int64_t(num_sms()) * 8;
  const int64_t blocks = ceil_div(vectors, kEwThreads);
  return unsigned(blocks < per_wave ? (blocks > 0 ? blocks : 1) : per_wave);
}

// ------------------------------------------------------------------ quantize --------------

template <typename T>
__global__ void __launch_bounds__(kEwThreads) quantize_kernel(QuantizeArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  const CastState cs = cast_begin(a.cast);
  const int64_t nvec = a.n / E;
  float amax = 0.0f;
  for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec;
       v += int64_t(gridDim.x) * blockDim.x) {
    float x[E];
    V::load(a.x, v * E, x);
#pragma unroll
    for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
    if (cs.store) cast_store<E>(a.out, v * E, x, cs);
  }
  block_amax_commit(amax, a.cast.amax_out);
}

// ------------------------------------------------------------------ register-resident -------
// act_lu and dact_dbias with each warp's rows of loads held in registers (the default path;
// the TMA-staged variants live in stream.cu).  Each CTA owns a strip of 32 x 16-byte column
// vectors and a chunk of rows; warps take rows in turn with several rows of loads in flight.

constexpr int kActWarps = 8;
constexpr int kActRows = 32;    // rows per CTA
constexpr int kActUnroll = 4;   // rows in flight per warp

// Each CTA owns a strip of 32 x 16-byte output vectors (one per lane) and kActRows rows; its
// warps take rows in turn, kActUnroll at a time, so every load is a 512-byte coalesced row
// segment and no index needs a division.
template <typename T>
__global__ void __launch_bounds__(kActWarps * 32, 3) act_lu_kernel(ActArgs a) {
  using V = Vec16<T>;
  using PR = Pairs<T>;
  constexpr int E = V::N;
  const CastState cs = cast_begin(a.cast);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool gated = a.act == TE_SWIGLU;
  const int64_t n_out = gated ? a.N_in / 2 : a.N_in;
  const int64_t col = (int64_t(blockIdx.x) * 32 + lane) * E;
  const int64_t r0 = int64_t(blockIdx.y) * kActRows;
  const int64_t r1 = r0 + kActRows < a.M ? r0 + kActRows : a.M;
  const T* x = static_cast<const T*>(a.x);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  float amax = 0.0f;
  if (col < n_out) {
    for (int64_t rb = r0 + warp; rb < r1; rb += kActUnroll * kActWarps) {
      uint4 rg[kActUnroll], rl[kActUnroll];
#pragma unroll
      for (int j = 0; j < kActUnroll; ++j) {
        const int64_t r = rb + int64_t(j) * kActWarps;
        const bool in = r < r1;
        rg[j] = in ? __ldg(reinterpret_cast<const uint4*>(x + r * a.N_in + col)) : zero;
        rl[j] = (in && gated) ? __ldg(reinterpret_cast<const uint4*>(x + r * a.N_in + n_out + col)) : zero;
      }
#pragma unroll
      for (int j = 0; j < kActUnroll; ++j) {
        const int64_t r = rb + int64_t(j) * kActWarps;
        if (r >= r1) break;
        f32x2 hp[PR::P], lp[PR::P];
        PR::get(rg[j], hp);
        if (gated) PR::get(rl[j], lp);
        float y[E];
#pragma unroll
        for (int p = 0; p < PR::P; ++p) {
          const f32x2 yy = gated ? mul2(silu2(hp[p]), lp[p]) : act2(a.act, hp[p]);
          amax = absmax2(amax, yy);
          y[2 * p] = f2lo(yy);
          y[2 * p + 1] = f2hi(yy);
        }
        if (cs.store) cast_store<E>(a.out, r * n_out + col, y, cs);
      }
    }
  }
  block_amax_commit(amax, a.cast.amax_out);
}

// ------------------------------------------------------------------ dact + dbias ----------

constexpr int kDactWarps = 8;
constexpr int kDactRows = 128;  // rows per CTA (chunk)

constexpr int kDactUnroll = 2;  // rows in flight per warp (x 24 warps per SM)

template <typename T>
__global__ void __launch_bounds__(kDactWarps * 32, 3) dact_dbias_kernel(DactArgs a) {
  using V = Vec16<T>;
  constexpr int E = V::N;
  constexpr int W = 32 * E;  // strip width in columns
  __shared__ float red[kDactWarps][2][W];
  const CastState cs = cast_begin(a.cast);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool gated = a.act == TE_SWIGLU;
  const bool ident = a.act == TE_IDENTITY;
  const int64_t n_out = gated ? a.N_in / 2 : a.N_in;
  const int64_t col = (int64_t(blockIdx.x) * 32 + lane) * E;
  const bool valid = col < n_out;
  const int64_t r0 = int64_t(blockIdx.y) * kDactRows;
  const int64_t r1 = r0 + kDactRows < a.M ? r0 + kDactRows : a.M;
  using PR = Pairs<T>;
  constexpr int P = PR::P;
  f32x2 acc1[P], acc2[P];
#pragma unroll
  for (int p = 0; p < P; ++p) { acc1[p] = f2s(0.0f); acc2[p] = f2s(0.0f); }
  float amax = 0.0f;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  if (valid) {
    for (int64_t rb = r0 + warp; rb < r1; rb += kDactUnroll * kDactWarps) {
      // issue every load of kDactUnroll rows before using any of them
      uint4 rdy[kDactUnroll], rx[kDactUnroll], rl[kDactUnroll];
#pragma unroll
      for (int j = 0; j < kDactUnroll; ++j) {
        const int64_t r = rb + int64_t(j) * kDactWarps;
        const bool in = r < r1;
        rdy[j] = in ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dy) + r * n_out + col)) : zero;
        rx[j] = (in && !ident) ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + r * a.N_in + col)) : zero;
        rl[j] = (in && gated) ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + r * a.N_in + n_out + col)) : zero;
      }
#pragma unroll
      for (int j = 0; j < kDactUnroll; ++j) {
        const int64_t r = rb + int64_t(j) * kDactWarps;
        if (r >= r1) break;
        f32x2 dyp[P], hp[P];
        PR::get(rdy[j], dyp);
        PR::get(rx[j], hp);
        if (gated) {
          f32x2 lp[P];
          PR::get(rl[j], lp);
          float dg[E], dl[E];
#pragma unroll
          for (int p = 0; p < P; ++p) {
            f32x2 sg, eg;
            sigmoid2(hp[p], sg, eg);
            // d_gate = dy * lin * silu'(gate), d_lin = dy * silu(gate)
            const f32x2 dsil = mul2(sg, fma2(hp[p], mul2(eg, sg), f2s(1.0f)));
            const f32x2 g2 = mul2(mul2(dyp[p], lp[p]), dsil);
            const f32x2 l2 = mul2(dyp[p], mul2(hp[p], sg));
            acc1[p] = add2(acc1[p], g2);
            acc2[p] = add2(acc2[p], l2);
            amax = absmax2(absmax2(amax, g2), l2);
            dg[2 * p] = f2lo(g2);
            dg[2 * p + 1] = f2hi(g2);
            dl[2 * p] = f2lo(l2);
            dl[2 * p + 1] = f2hi(l2);
          }
          if (cs.store) {
            cast_store<E>(a.dx, r * a.N_in + col, dg, cs);
            cast_store<E>(a.dx, r * a.N_in + n_out + col, dl, cs);
          }
        } else {
          float d[E];
#pragma unroll
          for (int p = 0; p < P; ++p) {
            const f32x2 dd = ident ? dyp[p] : mul2(dyp[p], dact2(a.act, hp[p]));
            acc1[p] = add2(acc1[p], dd);
            amax = absmax2(amax, dd);
            d[2 * p] = f2lo(dd);
            d[2 * p + 1] = f2hi(dd);
          }
          if (cs.store && a.dx) cast_store<E>(a.dx, r * a.N_in + col, d, cs);
        }
      }
    }
  }
  if (a.dbias) {
#pragma unroll
    for (int p = 0; p < P; ++p) {
      red[warp][0][lane * E + 2 * p] = f2lo(acc1[p]);
      red[warp][0][lane * E + 2 * p + 1] = f2hi(acc1[p]);
      red[warp][1][lane * E + 2 * p] = f2lo(acc2[p]);
      red[warp][1][lane * E + 2 * p + 1] = f2hi(acc2[p]);
    }
    __syncthreads();
    // 256 threads finish the strip's column sums, each over the 8 warps in warp order.
    const int halves = gated ? 2 : 1;
    for (int t = threadIdx.x; t < halves * W; t += blockDim.x) {
      const int hsel = t / W, j = t % W;
      float s = 0.0f;
#pragma unroll
      for (int w = 0; w < kDactWarps; ++w) s += red[w][hsel][j];
      const int64_t c = int64_t(blockIdx.x) * W + j;
      if (c < n_out) a.partials[int64_t(blockIdx.y) * a.N_in + hsel * n_out + c] = s;
    }
  }
  block_amax_commit(amax, a.cast.amax_out);
}

template <typename T>
te_status launch_dact_t(const DactArgs& a, cudaStream_t s) {
  constexpr int E = Vec16<T>::N;
  const int64_t n_out = a.act == TE_SWIGLU ? a.N_in / 2 : a.N_in;
  const int chunks = int(ceil_div(a.M, kDactRows));
  dim3 grid(unsigned(ceil_div(n_out, 32 * E)), unsigned(chunks));
  dact_dbias_kernel<T><<<grid, kDactWarps * 32, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

// ------------------------------------------------------------------ transpose -------------

// dst[C, R] = src[R, C]^T through a 32 x 33 shared tile (coalesced on both sides).
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float* src, int64_t R, int64_t C,
                                                            float* dst) {
  __shared__ float tile[32][33];
  const int64_t c0 = int64_t(blockIdx.x) * 32, r0 = int64_t(blockIdx.y) * 32;
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = src[r * C + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + threadIdx.x;
    if (c < C && r < R) dst[c * R + r] = tile[threadIdx.x][i];
  }
}

}  // namespace

te_status launch_act_lu_reg(const ActArgs& a, cudaStream_t s) {
  const int64_t n_out = a.act == TE_SWIGLU ? a.N_in / 2 : a.N_in;
  if (a.M == 0) return TE_OK;
  const int E = a.x_dtype == TE_BF16 ? 8 : 4;
  if (ceil_div(a.M, kActRows) > 65535) return TE_ERR_UNSUPPORTED;
  dim3 grid(unsigned(ceil_div(n_out, 32 * E)), unsigned(ceil_div(a.M, kActRows)));
  if (a.x_dtype == TE_BF16) {
    act_lu_kernel<__nv_bfloat16><<<grid, kActWarps * 32, 0, s>>>(a);
  } else if (a.x_dtype == TE_F32) {
    act_lu_kernel<float><<<grid, kActWarps * 32, 0, s>>>(a);
  } else {
    return TE_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

te_status launch_dact_reg(const DactArgs& a, cudaStream_t s) {
  if (a.dtype == TE_BF16) return launch_dact_t<__nv_bfloat16>(a, s);
  if (a.dtype == TE_F32) return launch_dact_t<float>(a, s);
  return TE_ERR_UNSUPPORTED;
}

te_status launch_transpose_f32(const float* src, int64_t R, int64_t C, float* dst, cudaStream_t s) {
  if (R == 0 || C == 0) return TE_OK;
  if (ceil_div(R, 32) > 65535) return TE_ERR_UNSUPPORTED;
  ProfileScope prof(TE_KERNEL_TRANSPOSE, s);
  dim3 grid(unsigned(ceil_div(C, 32)), unsigned(ceil_div(R, 32)));
  transpose_f32_kernel<<<grid, dim3(32, 8), 0, s>>>(src, R, C, dst);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

te_status launch_quantize(const QuantizeArgs& a, cudaStream_t s) {
  ProfileScope prof(TE_KERNEL_QUANTIZE, s);
  if (a.x_dtype == TE_BF16) {
    quantize_kernel<__nv_bfloat16><<<ew_grid(a.n / 8), kEwThreads, 0, s>>>(a);
  } else if (a.x_dtype == TE_F32) {
    quantize_kernel<float><<<ew_grid(a.n / 4), kEwThreads, 0, s>>>(a);
  } else {
    return TE_ERR_UNSUPPORTED;
  }
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

}  // namespace te
