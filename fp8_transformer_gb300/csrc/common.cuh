// Device helpers shared by the kernels of the fused norm + feed-forward block (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "te_gb300.h"

namespace te {

constexpr float kE4M3Max = 448.0f;

// ------------------------------------------------------------------ conversions ------------

// Two fp32 -> two bf16 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Two fp32 -> two E4M3 bytes, round to nearest even, saturating to +-448 (satfinite).
// `lo` lands in the low byte.
__device__ __forceinline__ uint16_t pack_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four fp32 -> four E4M3 bytes (element 0 in the lowest byte).
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  return uint32_t(pack_e4m3x2(a, b)) | (uint32_t(pack_e4m3x2(c, d)) << 16);
}

// Two E4M3 bytes -> two exact fp32 values (via the exact E4M3 -> f16 conversion).
__device__ __forceinline__ float2 unpack_e4m3x2(uint16_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// ------------------------------------------------------------------ packed fp32 pairs -----
// sm_100+ executes two IEEE fp32 operations per f32x2 instruction (round to nearest, no
// flush-to-zero); the bandwidth-bound kernels run their arithmetic on such pairs.

using f32x2 = float2;

__device__ __forceinline__ f32x2 f2(float lo, float hi) { return make_float2(lo, hi); }
__device__ __forceinline__ f32x2 f2s(float v) { return make_float2(v, v); }
__device__ __forceinline__ float f2lo(f32x2 v) { return v.x; }
__device__ __forceinline__ float f2hi(f32x2 v) { return v.y; }
__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) { return __ffma2_rn(a, b, c); }
// a - b, rounded once (b * -1 is exact).
__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) { return __ffma2_rn(b, f2s(-1.0f), a); }
// bf16x2 word -> fp32 pair (exact).
__device__ __forceinline__ f32x2 bf16x2_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ float absmax2(float m, f32x2 v) {
  return fmaxf(m, fmaxf(fabsf(v.x), fabsf(v.y)));
}

// ------------------------------------------------------------------ activations -----------
// Written from their definitions, in fp32.  The tanh-form GELU uses the identity
// 0.5 * (1 + tanh(u)) = 1 / (1 + exp(-2u)), which is the same function but avoids the
// cancellation of 1 + tanh(u) for negative u; likewise 1 - tanh(u)^2 = 4 s(2u) s(-2u) with
// s the logistic function, and 1 - s(z) = exp(-z) s(z).

constexpr float kGeluK0 = 0.7978845608028654f;  // sqrt(2 / pi)
constexpr float kGeluK1 = 0.044715f;

__device__ __forceinline__ float gelu_u(float h) { return kGeluK0 * (h + kGeluK1 * h * h * h); }

__device__ __forceinline__ float act_gelu(float h) {
  return h / (1.0f + expf(-2.0f * gelu_u(h)));
}

__device__ __forceinline__ float act_silu(float z) { return z / (1.0f + expf(-z)); }

__device__ __forceinline__ float act_relu(float h) { return h > 0.0f ? h : 0.0f; }

// silu'(z) = s (1 + z (1 - s)), s = 1 / (1 + exp(-z)), with 1 - s = exp(-z) s.
__device__ __forceinline__ float dsilu(float z) {
  const float e = expf(-fmaxf(z, -80.0f));
  const float s = 1.0f / (1.0f + e);
  return s * (1.0f + z * (e * s));
}

// gelu'(h) = 0.5 (1 + t) + 0.5 h (1 - t^2) sqrt(2/pi) (1 + 3 * 0.044715 h^2), t = tanh(u),
// evaluated as sp + 2 h sqrt(2/pi) (1 + 3 * 0.044715 h^2) sp sn with sp = s(2u), sn = s(-2u).
__device__ __forceinline__ float dgelu(float h) {
  const float u = gelu_u(h);
  const float e = expf(-2.0f * fmaxf(u, -40.0f));
  const float sp = 1.0f / (1.0f + e);
  const float sn = e * sp;
  return sp + 2.0f * h * kGeluK0 * (1.0f + 3.0f * kGeluK1 * h * h) * sp * sn;
}

// Bandwidth-bound kernels evaluate the derivatives with the hardware exp2 / reciprocal
// approximations (relative error ~1e-6), so that arithmetic stays under the memory time.
__device__ __forceinline__ float fast_rcp(float x) { return __fdividef(1.0f, x); }

__device__ __forceinline__ float silu_fast(float z) { return z * fast_rcp(1.0f + __expf(-z)); }

__device__ __forceinline__ float dsilu_fast(float z) {
  const float e = __expf(-fmaxf(z, -80.0f));
  const float s = fast_rcp(1.0f + e);
  return s * (1.0f + z * (e * s));
}

__device__ __forceinline__ float dgelu_fast(float h) {
  const float u = gelu_u(h);
  const float e = __expf(-2.0f * fmaxf(u, -40.0f));
  const float sp = fast_rcp(1.0f + e);
  const float sn = e * sp;
  return sp + 2.0f * h * kGeluK0 * (1.0f + 3.0f * kGeluK1 * h * h) * sp * sn;
}

__device__ __forceinline__ float gelu_fast(float h) {
  return h * fast_rcp(1.0f + __expf(-2.0f * gelu_u(h)));
}

__device__ __forceinline__ float act_fast(int act, float h) {
  switch (act) {
    case TE_RELU: return act_relu(h);
    case TE_GELU: return gelu_fast(h);
    case TE_SILU: return silu_fast(h);
    default: return h;
  }
}

// Pairwise versions for the bandwidth-bound kernels.  exp(x) = 2^(x log2 e) on the hardware
// exp2 approximation, 1/x on the hardware reciprocal approximation; arguments are clamped so
// that no exp2 result overflows where a product with it follows.
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
__device__ __forceinline__ f32x2 ex2_2(f32x2 a) {
  return f2(ex2_approx(f2lo(a)), ex2_approx(f2hi(a)));
}
__device__ __forceinline__ f32x2 rcp2(f32x2 a) {
  return f2(rcp_approx(f2lo(a)), rcp_approx(f2hi(a)));
}
__device__ __forceinline__ f32x2 min2s(f32x2 a, float m) {
  return f2(fminf(f2lo(a), m), fminf(f2hi(a), m));
}

// logistic s(z) = 1 / (1 + exp(-z)) and e = exp(-z), with z clamped at -80 inside exp.
__device__ __forceinline__ void sigmoid2(f32x2 z, f32x2& s, f32x2& e) {
  e = ex2_2(min2s(mul2(z, f2s(-kLog2e)), 80.0f * kLog2e));
  s = rcp2(add2(e, f2s(1.0f)));
}

// -2 u log2(e) with u = sqrt(2/pi) (h + 0.044715 h^3), as h (c1 + c2 h^2).
constexpr float kGeluA1 = -2.0f * kLog2e * kGeluK0;
constexpr float kGeluA2 = -2.0f * kLog2e * kGeluK0 * kGeluK1;

// gelu(h) = h s(2u) = h / (1 + 2^(-2u log2 e)); an infinite exp2 gives the correct limit 0.
__device__ __forceinline__ f32x2 gelu2(f32x2 h) {
  const f32x2 a = mul2(h, fma2(mul2(h, h), f2s(kGeluA2), f2s(kGeluA1)));
  return mul2(h, rcp2(add2(ex2_2(a), f2s(1.0f))));
}

// gelu'(h) = s + 2 h sqrt(2/pi) (1 + 3 * 0.044715 h^2) s (1 - s), s = logistic(2u),
// 1 - s = e s with e = exp(-2u) (the exponent is clamped so e stays finite).
__device__ __forceinline__ f32x2 dgelu2(f32x2 h) {
  const f32x2 hh = mul2(h, h);
  const f32x2 a = min2s(mul2(h, fma2(hh, f2s(kGeluA2), f2s(kGeluA1))), 80.0f * kLog2e);
  const f32x2 e = ex2_2(a);
  const f32x2 s = rcp2(add2(e, f2s(1.0f)));
  const f32x2 q = mul2(h, fma2(hh, f2s(6.0f * kGeluK0 * kGeluK1), f2s(2.0f * kGeluK0)));
  return fma2(q, mul2(s, mul2(e, s)), s);
}

// silu(z) = z / (1 + 2^(-z log2 e)); an infinite exp2 gives the correct limit 0.
__device__ __forceinline__ f32x2 silu2(f32x2 z) {
  return mul2(z, rcp2(add2(ex2_2(mul2(z, f2s(-kLog2e))), f2s(1.0f))));
}

// silu'(z) = s (1 + z (1 - s)).
__device__ __forceinline__ f32x2 dsilu2(f32x2 z) {
  f32x2 s, e;
  sigmoid2(z, s, e);
  return mul2(s, fma2(z, mul2(e, s), f2s(1.0f)));
}

__device__ __forceinline__ f32x2 relu2(f32x2 h) {
  return f2(fmaxf(f2lo(h), 0.0f), fmaxf(f2hi(h), 0.0f));
}
__device__ __forceinline__ f32x2 drelu2(f32x2 h) {
  return f2(f2lo(h) > 0.0f ? 1.0f : 0.0f, f2hi(h) > 0.0f ? 1.0f : 0.0f);
}

// Compile-time activation choice (the inner loops are instantiated per activation).
template <int ACT>
__device__ __forceinline__ f32x2 act2c(f32x2 h) {
  if constexpr (ACT == TE_RELU) return relu2(h);
  else if constexpr (ACT == TE_GELU) return gelu2(h);
  else if constexpr (ACT == TE_SILU) return silu2(h);
  else return h;
}
template <int ACT>
__device__ __forceinline__ f32x2 dact2c(f32x2 h) {
  if constexpr (ACT == TE_RELU) return drelu2(h);
  else if constexpr (ACT == TE_GELU) return dgelu2(h);
  else if constexpr (ACT == TE_SILU) return dsilu2(h);
  else return f2s(1.0f);
}

__device__ __forceinline__ f32x2 act2(int act, f32x2 h) {
  switch (act) {
    case TE_RELU: return relu2(h);
    case TE_GELU: return gelu2(h);
    case TE_SILU: return silu2(h);
    default: return h;
  }
}
__device__ __forceinline__ f32x2 dact2(int act, f32x2 h) {
  switch (act) {
    case TE_RELU: return drelu2(h);
    case TE_GELU: return dgelu2(h);
    case TE_SILU: return dsilu2(h);
    default: return f2s(1.0f);
  }
}

__device__ __forceinline__ float dact_fast(int act, float h) {
  switch (act) {
    case TE_RELU: return h > 0.0f ? 1.0f : 0.0f;
    case TE_GELU: return dgelu_fast(h);
    case TE_SILU: return dsilu_fast(h);
    default: return 1.0f;
  }
}

// Non-gated activation by id (TE_IDENTITY, TE_RELU, TE_GELU, TE_SILU).
__device__ __forceinline__ float act_apply(int act, float h) {
  switch (act) {
    case TE_RELU: return act_relu(h);
    case TE_GELU: return act_gelu(h);
    case TE_SILU: return act_silu(h);
    default: return h;
  }
}

// d/dh of the non-gated activations.
__device__ __forceinline__ float dact_apply(int act, float h) {
  switch (act) {
    case TE_RELU: return h > 0.0f ? 1.0f : 0.0f;
    case TE_GELU: return dgelu(h);
    case TE_SILU: return dsilu(h);
    default: return 1.0f;
  }
}

// ------------------------------------------------------------------ scaling ---------------

// scale = 448 / amax; 1 when amax is 0 or not finite; FLT_MAX when the quotient overflows.
__device__ __forceinline__ float scale_from_amax(float amax) {
  if (!(amax > 0.0f) || !isfinite(amax)) return 1.0f;
  float s = kE4M3Max / amax;
  if (!isfinite(s)) s = 3.4028234663852886e38f;
  return s;
}

// ------------------------------------------------------------------ reductions ------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// amax of non-negative floats: their bit patterns order like the values.
__device__ __forceinline__ void atomic_max_nonneg(float* addr, float v) {
  if (v > 0.0f) atomicMax(reinterpret_cast<int*>(addr), __float_as_int(v));
}

// Block-wide max of a per-thread value, then one atomic per block (blockDim.x <= 1024).
__device__ __forceinline__ void block_amax_commit(float v, float* amax) {
  __shared__ float red[32];
  v = warp_max(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = v;
  __syncthreads();
  if (w == 0) {
    const int nw = (blockDim.x + 31) >> 5;
    float m = l < nw ? red[l] : 0.0f;
    m = warp_max(m);
    if (l == 0 && amax) atomic_max_nonneg(amax, m);
  }
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace te
