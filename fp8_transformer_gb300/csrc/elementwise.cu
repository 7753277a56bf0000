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
