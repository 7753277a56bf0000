// Bandwidth-bound kernels of the block: per-tensor quantize, activation, the backward's fused
// activation gradient + bias reduction + quantize, and the fp32 transpose of the tf32 path.
//
// * quantize (TransformerEngine JAX "LayerNorm Dense" page, Description: the normalized output
//   and the kernel are quantized before the GEMM): 16-byte vectors, grid-stride, amax by one
//   integer atomic per block.
// * act_lu ("Activation" page, Description: the forward rule's activation primitive, optional
//   FP8 round trip) and dact_dbias ("LayerNorm MLP" page, Description, backward: the fused
//   quantize / dact / dbias primitive).  Each CTA owns a strip of 32 x 16-byte column vectors
//   (one per lane) and a chunk of rows; its warps take rows in turn with several rows of loads
//   in flight, so every access is a 512-byte coalesced row segment and no index needs a
//   division.  The activation and the output kind are compile-time choices of the inner loop,
//   and the arithmetic runs on f32x2 pairs with the hardware exp2 / reciprocal.  For dbias
//   every thread sums its columns over the chunk in registers, the 8 warps of the CTA combine
//   through shared memory in warp order, one partial row per chunk goes to the workspace, and
//   a second kernel adds the partial rows in chunk order, so dbias is deterministic.
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
  // the kernel after this one may launch its setup now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using V = Vec16<T>;
  constexpr int E = V::N;
  const CastState cs = cast_begin(a.cast);
  const int64_t nvec = a.n / E;
  float amax = 0.0f;
  with_out(out_kind(cs), [&](auto tag) {
    constexpr int OUT = decltype(tag)::value;
    for (int64_t v = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; v < nvec;
         v += int64_t(gridDim.x) * blockDim.x) {
      float x[E];
      V::load(a.x, v * E, x);
#pragma unroll
      for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
      store_out<OUT, E>(a.out, v * E, x, cs);
    }
  });
  block_amax_commit(amax, a.cast.amax_out);
}

// ------------------------------------------------------------------ act_lu ----------------

constexpr int kActWarps = 8;
constexpr int kActRows = 32;    // rows per CTA
constexpr int kActUnroll = 4;   // rows in flight per warp

template <typename T, int ACT>
__global__ void __launch_bounds__(kActWarps * 32, 3) act_lu_kernel(ActArgs a) {
  // the kernel after this one may launch its setup now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using PR = Pairs<T>;
  constexpr int E = Vec16<T>::N;
  constexpr bool kGated = is_gated(ACT);
  constexpr int kBase = gate_act(ACT);  // the function of the gate half
  const CastState cs = cast_begin(a.cast);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n_out = kGated ? a.N_in / 2 : a.N_in;
  const int64_t col = (int64_t(blockIdx.x) * 32 + lane) * E;
  const int64_t r0 = int64_t(blockIdx.y) * kActRows;
  const int64_t r1 = r0 + kActRows < a.M ? r0 + kActRows : a.M;
  const T* x = static_cast<const T*>(a.x);
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const bool want_amax = a.cast.amax_out != nullptr;
  float am[PR::P];  // one running amax per pair position: no single long chain
#pragma unroll
  for (int p = 0; p < PR::P; ++p) am[p] = 0.0f;
  if (col < n_out) {
    with_out_amax(out_kind(cs), want_amax, [&](auto tag, auto atag) {
      constexpr int OUT = decltype(tag)::value;
      constexpr bool AMAX = decltype(atag)::value;
      for (int64_t rb = r0 + warp; rb < r1; rb += kActUnroll * kActWarps) {
        uint4 rg[kActUnroll], rl[kActUnroll];  // rl: the linear halves (gated types only)
        (void)rl;
#pragma unroll
        for (int j = 0; j < kActUnroll; ++j) {
          const int64_t r = rb + int64_t(j) * kActWarps;
          const bool in = r < r1;
          rg[j] = in ? __ldg(reinterpret_cast<const uint4*>(x + r * a.N_in + col)) : zero;
          if constexpr (kGated)
            rl[j] = in ? __ldg(reinterpret_cast<const uint4*>(x + r * a.N_in + n_out + col)) : zero;
        }
#pragma unroll
        for (int j = 0; j < kActUnroll; ++j) {
          const int64_t r = rb + int64_t(j) * kActWarps;
          if (r >= r1) break;
          f32x2 hp[PR::P], lp[PR::P];
          (void)lp;
          PR::get(rg[j], hp);
          if constexpr (kGated) PR::get(rl[j], lp);
          float y[E];
#pragma unroll
          for (int p = 0; p < PR::P; ++p) {
            f32x2 yy;
            if constexpr (kGated) yy = mul2(act2c<kBase>(hp[p]), lp[p]);
            else yy = act2c<ACT>(hp[p]);
            if (AMAX) am[p] = absmax2(am[p], yy);
            y[2 * p] = f2lo(yy);
            y[2 * p + 1] = f2hi(yy);
          }
          store_out<OUT, E>(a.out, r * n_out + col, y, cs);
        }
      }
    });
  }
  float amax = am[0];
#pragma unroll
  for (int p = 1; p < PR::P; ++p) amax = fmaxf(amax, am[p]);
  block_amax_commit(amax, a.cast.amax_out);
}

// ------------------------------------------------------------------ dact + dbias ----------

constexpr int kDactWarps = 8;
constexpr int kDactRows = 128;  // rows per CTA (chunk) = rows per dbias partial
constexpr int kDactUnroll = 2;  // rows in flight per warp (twice that when only dy is read)

// (three CTAs per SM; two for a gated pair, whose third input row per load would not fit the
// register budget of three)
template <typename T, int ACT>
__global__ void __launch_bounds__(kDactWarps * 32, is_gated(ACT) ? 2 : 3)
    dact_dbias_kernel(DactArgs a) {
  using PR = Pairs<T>;
  constexpr int E = Vec16<T>::N;
  constexpr int P = PR::P;
  constexpr int W = 32 * E;  // strip width in columns
  constexpr bool kGated = is_gated(ACT);
  constexpr int kBase = gate_act(ACT);  // the function of the gate half
  constexpr bool kIdent = ACT == TE_IDENTITY;
  // rows whose loads are in flight at once per warp: with the identity only dy is read, so
  // twice as many rows keep as many bytes in flight
  constexpr int U = kIdent ? 2 * kDactUnroll : kDactUnroll;
  __shared__ float red[kDactWarps][2][W];
  // the column-sum kernel that follows may launch now: it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const CastState cs = cast_begin(a.cast);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n_out = kGated ? a.N_in / 2 : a.N_in;
  const int64_t col = (int64_t(blockIdx.x) * 32 + lane) * E;
  const int64_t r0 = int64_t(blockIdx.y) * kDactRows;
  const int64_t r1 = r0 + kDactRows < a.M ? r0 + kDactRows : a.M;
  f32x2 acc1[P], acc2[P];
#pragma unroll
  for (int p = 0; p < P; ++p) { acc1[p] = f2s(0.0f); acc2[p] = f2s(0.0f); }
  float am[P];  // one running amax per pair position: no single long chain
#pragma unroll
  for (int p = 0; p < P; ++p) am[p] = 0.0f;
  const bool want_amax = a.cast.amax_out != nullptr;
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  if (col < n_out) {
    with_out_amax(a.dx ? out_kind(cs) : int(OUT_NONE), want_amax, [&](auto tag, auto atag) {
      constexpr int OUT = decltype(tag)::value;
      constexpr bool AMAX = decltype(atag)::value;
      for (int64_t rb = r0 + warp; rb < r1; rb += U * kDactWarps) {
        // every load of U rows is issued before any of them is used
        uint4 rdy[U], rx[U], rl[U];  // rx, rl unused by some types
        (void)rx;
        (void)rl;
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int64_t r = rb + int64_t(j) * kDactWarps;
          const bool in = r < r1;
          rdy[j] = in ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.dy) + r * n_out + col)) : zero;
          if constexpr (!kIdent)
            rx[j] = in ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + r * a.N_in + col)) : zero;
          if constexpr (kGated)
            rl[j] = in ? __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(a.x) + r * a.N_in + n_out + col)) : zero;
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
          const int64_t r = rb + int64_t(j) * kDactWarps;
          if (r >= r1) break;
          f32x2 dyp[P], hp[P];
          (void)hp;
          PR::get(rdy[j], dyp);
          if constexpr (!kIdent) PR::get(rx[j], hp);
          if constexpr (kGated) {
            f32x2 lp[P];
            PR::get(rl[j], lp);
            float dg[E], dl[E];
#pragma unroll
            for (int p = 0; p < P; ++p) {
              // d_gate = dy * lin * base'(gate), d_lin = dy * base(gate)
              f32x2 act_g, dact_g;
              if constexpr (kBase == TE_SILU) {  // silu and silu' share one logistic
                f32x2 sg, eg;
                sigmoid2(hp[p], sg, eg);
                dact_g = mul2(sg, fma2(hp[p], mul2(eg, sg), f2s(1.0f)));
                act_g = mul2(hp[p], sg);
              } else {
                act_g = act2c<kBase>(hp[p]);
                dact_g = dact2c<kBase>(hp[p]);
              }
              const f32x2 g2 = mul2(mul2(dyp[p], lp[p]), dact_g);
              const f32x2 l2 = mul2(dyp[p], act_g);
              acc1[p] = add2(acc1[p], g2);
              acc2[p] = add2(acc2[p], l2);
              if (AMAX) am[p] = absmax2(absmax2(am[p], g2), l2);
              dg[2 * p] = f2lo(g2);
              dg[2 * p + 1] = f2hi(g2);
              dl[2 * p] = f2lo(l2);
              dl[2 * p + 1] = f2hi(l2);
            }
            store_out<OUT, E>(a.dx, r * a.N_in + col, dg, cs);
            store_out<OUT, E>(a.dx, r * a.N_in + n_out + col, dl, cs);
          } else {
            float d[E];
#pragma unroll
            for (int p = 0; p < P; ++p) {
              f32x2 dd;
              if constexpr (kIdent) dd = dyp[p];
              else dd = mul2(dyp[p], dact2c<ACT>(hp[p]));
              acc1[p] = add2(acc1[p], dd);
              if (AMAX) am[p] = absmax2(am[p], dd);
              d[2 * p] = f2lo(dd);
              d[2 * p + 1] = f2hi(dd);
            }
            store_out<OUT, E>(a.dx, r * a.N_in + col, d, cs);
          }
        }
      }
    });
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
    // the CTA's threads finish the strip's column sums, each over the 8 warps in warp order
    const int halves = kGated ? 2 : 1;
    for (int t = threadIdx.x; t < halves * W; t += blockDim.x) {
      const int hsel = t / W, j = t % W;
      float sum = 0.0f;
#pragma unroll
      for (int w = 0; w < kDactWarps; ++w) sum += red[w][hsel][j];
      const int64_t c = int64_t(blockIdx.x) * W + j;
      if (c < n_out) a.partials[int64_t(blockIdx.y) * a.N_in + hsel * n_out + c] = sum;
    }
  }
  float amax = am[0];
#pragma unroll
  for (int p = 1; p < P; ++p) amax = fmaxf(amax, am[p]);
  block_amax_commit(amax, a.cast.amax_out);
}

// out[j] = sum_c partials[c][j] (n a multiple of 4), summed in the same order for every column
// and every run: a CTA takes 128 columns, 4 per thread of a warp (16-byte loads); its warps take
// the chunks c = w, w + kColsumWarps, ... each in chunk order, and the warps' sums are then
// added in warp order.  (One thread per column looping over every chunk was a chain of ~128
// dependent loads.)
constexpr int kColsumWarps = 16;
__global__ void __launch_bounds__(kColsumWarps * 32)
    colsum_partials_kernel(const float* partials, int chunks, int64_t n, float* out) {
  __shared__ float4 sums[kColsumWarps][32];
  // launched as a programmatic dependent of the dact kernel: wait for that grid's partials
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t j = int64_t(blockIdx.x) * 128 + lane * 4;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  if (j < n) {
#pragma unroll 4
    for (int c = w; c < chunks; c += kColsumWarps) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(partials + int64_t(c) * n + j));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
  }
  sums[w][lane] = acc;
  __syncthreads();
  if (w == 0 && j < n) {
    float4 t = sums[0][lane];
#pragma unroll
    for (int v = 1; v < kColsumWarps; ++v) {
      const float4 u = sums[v][lane];
      t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
    }
    out[j] = t.x; out[j + 1] = t.y; out[j + 2] = t.z; out[j + 3] = t.w;
  }
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

template <typename T>
te_status launch_act_t(const ActArgs& a, dim3 grid, cudaStream_t s) {
  switch (a.act) {
    case TE_RELU: act_lu_kernel<T, TE_RELU><<<grid, kActWarps * 32, 0, s>>>(a); break;
    case TE_GELU: act_lu_kernel<T, TE_GELU><<<grid, kActWarps * 32, 0, s>>>(a); break;
    case TE_SILU: act_lu_kernel<T, TE_SILU><<<grid, kActWarps * 32, 0, s>>>(a); break;
    case TE_SWIGLU: act_lu_kernel<T, TE_SWIGLU><<<grid, kActWarps * 32, 0, s>>>(a); break;
    case TE_GEGLU: act_lu_kernel<T, TE_GEGLU><<<grid, kActWarps * 32, 0, s>>>(a); break;
    case TE_REGLU: act_lu_kernel<T, TE_REGLU><<<grid, kActWarps * 32, 0, s>>>(a); break;
    default: act_lu_kernel<T, TE_IDENTITY><<<grid, kActWarps * 32, 0, s>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T>
te_status launch_dact_t(const DactArgs& a, dim3 grid, cudaStream_t s) {
  switch (a.act) {
    case TE_RELU: dact_dbias_kernel<T, TE_RELU><<<grid, kDactWarps * 32, 0, s>>>(a); break;
    case TE_GELU: dact_dbias_kernel<T, TE_GELU><<<grid, kDactWarps * 32, 0, s>>>(a); break;
    case TE_SILU: dact_dbias_kernel<T, TE_SILU><<<grid, kDactWarps * 32, 0, s>>>(a); break;
    case TE_SWIGLU: dact_dbias_kernel<T, TE_SWIGLU><<<grid, kDactWarps * 32, 0, s>>>(a); break;
    case TE_GEGLU: dact_dbias_kernel<T, TE_GEGLU><<<grid, kDactWarps * 32, 0, s>>>(a); break;
    case TE_REGLU: dact_dbias_kernel<T, TE_REGLU><<<grid, kDactWarps * 32, 0, s>>>(a); break;
    default: dact_dbias_kernel<T, TE_IDENTITY><<<grid, kDactWarps * 32, 0, s>>>(a); break;
  }
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

}  // namespace

te_status launch_act_lu(const ActArgs& a, cudaStream_t s) {
  ProfileScope prof(TE_KERNEL_ACT_LU, s);
  if (a.M == 0) return TE_OK;
  const int64_t n_out = is_gated(a.act) ? a.N_in / 2 : a.N_in;
  const int E = a.x_dtype == TE_BF16 ? 8 : 4;
  if (ceil_div(a.M, kActRows) > 65535) return TE_ERR_UNSUPPORTED;
  dim3 grid(unsigned(ceil_div(n_out, 32 * E)), unsigned(ceil_div(a.M, kActRows)));
  if (a.x_dtype == TE_BF16) return launch_act_t<__nv_bfloat16>(a, grid, s);
  if (a.x_dtype == TE_F32) return launch_act_t<float>(a, grid, s);
  return TE_ERR_UNSUPPORTED;
}

size_t dact_dbias_workspace(int64_t M, int64_t N_in) {
  return size_t(ceil_div(M > 0 ? M : 1, kDactRows)) * size_t(N_in) * sizeof(float);
}

te_status launch_dact_dbias(const DactArgs& a, cudaStream_t s) {
  if (a.M == 0) return TE_OK;
  ProfileScope prof(TE_KERNEL_DACT_DBIAS, s);
  const int64_t n_out = is_gated(a.act) ? a.N_in / 2 : a.N_in;
  const int E = a.dtype == TE_BF16 ? 8 : 4;
  const int chunks = int(ceil_div(a.M, kDactRows));
  if (chunks > 65535) return TE_ERR_UNSUPPORTED;
  dim3 grid(unsigned(ceil_div(n_out, 32 * E)), unsigned(chunks));
  te_status st = a.dtype == TE_BF16 ? launch_dact_t<__nv_bfloat16>(a, grid, s)
                 : a.dtype == TE_F32 ? launch_dact_t<float>(a, grid, s)
                                     : TE_ERR_UNSUPPORTED;
  if (st != TE_OK || !a.dbias) return st;
  return launch_dependent(colsum_partials_kernel, dim3(unsigned(ceil_div(a.N_in, 128))),
                          dim3(kColsumWarps * 32), s, static_cast<const float*>(a.partials),
                          chunks, int64_t(a.N_in), a.dbias);
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

// ------------------------------------------------------------------ scale update ---------

__global__ void update_scales_kernel(ScaleUpdateArgs a) {
  const int i = threadIdx.x;
  if (i >= a.n) return;
  const float s = scale_from_amax(*a.amax[i]);
  *a.scale[i] = s;
  if (a.scale_inv[i]) *a.scale_inv[i] = 1.0f / s;
}

te_status launch_update_scales(const ScaleUpdateArgs& a, cudaStream_t s) {
  if (a.n <= 0) return TE_OK;
  update_scales_kernel<<<1, 32, 0, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

}  // namespace te
