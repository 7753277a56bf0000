// Output stage of the bandwidth-bound kernels: fp32 results -> fp32 / bf16 / E4M3 storage,
// with the per-tensor amax and scale bookkeeping.
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace te {

struct CastState {
  float scale = 1.0f;
  float scale_inv = 1.0f;
  int out_dtype = TE_BF16;
  int fake_quant = 0;
  int store = 1;
};

// Reads the scale (given, or derived from this call's amax); the first thread of the grid
// publishes scale / scale_inv when the pass stores.
__device__ __forceinline__ CastState cast_begin(const CastSpec& c) {
  CastState s;
  s.out_dtype = c.out_dtype;
  s.fake_quant = c.fake_quant;
  s.store = c.store;
  if (c.out_dtype == TE_E4M3 || c.fake_quant) {
    if (c.amax_in) s.scale = scale_from_amax(*c.amax_in);
    else if (c.scale) s.scale = *c.scale;
    s.scale_inv = 1.0f / s.scale;
  }
  if (c.store && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && threadIdx.y == 0) {
    if (c.scale_out) *c.scale_out = s.scale;
    if (c.scale_inv_out) *c.scale_inv_out = s.scale_inv;
  }
  return s;
}

// E4M3 round trip of one value: fp32(decode(E4M3(fp32(v * scale))) * scale_inv).
__device__ __forceinline__ float fake_quant1(float v, float scale, float scale_inv) {
  float2 d = unpack_e4m3x2(pack_e4m3x2(v * scale, 0.0f));
  return d.x * scale_inv;
}

// Output kinds, chosen once per kernel (outside every per-element loop) so that each inner
// loop is compiled for exactly one kind.
enum OutKind : int {
  OUT_F32 = 0,
  OUT_BF16 = 1,
  OUT_E4M3 = 2,
  OUT_FAKE_F32 = 3,   // E4M3 round trip stored as fp32
  OUT_FAKE_BF16 = 4,  // E4M3 round trip stored as bf16
  OUT_NONE = 5        // amax pass of current scaling: nothing stored
};

__host__ __device__ __forceinline__ int out_kind_of(int store, int out_dtype, int fake_quant) {
  if (!store) return OUT_NONE;
  if (out_dtype == TE_E4M3) return OUT_E4M3;
  if (fake_quant) return out_dtype == TE_F32 ? OUT_FAKE_F32 : OUT_FAKE_BF16;
  return out_dtype == TE_F32 ? OUT_F32 : OUT_BF16;
}

__device__ __forceinline__ int out_kind(const CastState& cs) {
  return out_kind_of(cs.store, cs.out_dtype, cs.fake_quant);
}

template <int K>
struct OutTag {
  static constexpr int value = K;
};

// Calls f(OutTag<kind>{}) with the kind as a compile-time constant.
template <class F>
__device__ __forceinline__ void with_out(int kind, F&& f) {
  switch (kind) {
    case OUT_F32: f(OutTag<OUT_F32>{}); break;
    case OUT_BF16: f(OutTag<OUT_BF16>{}); break;
    case OUT_E4M3: f(OutTag<OUT_E4M3>{}); break;
    case OUT_FAKE_F32: f(OutTag<OUT_FAKE_F32>{}); break;
    case OUT_FAKE_BF16: f(OutTag<OUT_FAKE_BF16>{}); break;
    default: f(OutTag<OUT_NONE>{}); break;
  }
}

template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

// Calls f(OutTag<kind>{}, BoolTag<amax>{}) with both as compile-time constants (inside a kernel,
// or on the host to pick a kernel compiled for one kind).  The kinds that quantize or only
// measure always take the amax (their callers always ask for it); plain fp32 / bf16 stores take
// it when `want_amax`.
#pragma nv_exec_check_disable
template <class F>
__host__ __device__ __forceinline__ void with_out_amax(int kind, bool want_amax, F&& f) {
  switch (kind) {
    case OUT_F32:
      if (want_amax) f(OutTag<OUT_F32>{}, BoolTag<true>{});
      else f(OutTag<OUT_F32>{}, BoolTag<false>{});
      break;
    case OUT_BF16:
      if (want_amax) f(OutTag<OUT_BF16>{}, BoolTag<true>{});
      else f(OutTag<OUT_BF16>{}, BoolTag<false>{});
      break;
    case OUT_E4M3: f(OutTag<OUT_E4M3>{}, BoolTag<true>{}); break;
    case OUT_FAKE_F32: f(OutTag<OUT_FAKE_F32>{}, BoolTag<true>{}); break;
    case OUT_FAKE_BF16: f(OutTag<OUT_FAKE_BF16>{}, BoolTag<true>{}); break;
    default: f(OutTag<OUT_NONE>{}, BoolTag<true>{}); break;
  }
}

// Stores N (4 or 8) consecutive values at element index `idx` (a multiple of N) of `out`.
template <int OUT, int N>
__device__ __forceinline__ void store_out(void* out, int64_t idx, const float (&y)[N],
                                          const CastState& cs) {
  static_assert(N == 4 || N == 8, "vector of 4 or 8");
  if constexpr (OUT == OUT_NONE) {
    return;
  } else if constexpr (OUT == OUT_E4M3) {
    const f32x2 s2 = f2s(cs.scale);
    uint32_t w[N / 4];
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
      const f32x2 a = mul2(f2(y[4 * i], y[4 * i + 1]), s2);
      const f32x2 b = mul2(f2(y[4 * i + 2], y[4 * i + 3]), s2);
      w[i] = pack_e4m3x4(f2lo(a), f2hi(a), f2lo(b), f2hi(b));
    }
    uint8_t* base = static_cast<uint8_t*>(out) + idx;
    if constexpr (N == 8) {
      *reinterpret_cast<uint2*>(base) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t*>(base) = w[0];
    }
  } else {
    float v[N];
#pragma unroll
    for (int i = 0; i < N; ++i)
      v[i] = (OUT == OUT_FAKE_F32 || OUT == OUT_FAKE_BF16) ? fake_quant1(y[i], cs.scale, cs.scale_inv)
                                                          : y[i];
    if constexpr (OUT == OUT_F32 || OUT == OUT_FAKE_F32) {
      float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
      p[0] = make_float4(v[0], v[1], v[2], v[3]);
      if constexpr (N == 8) p[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      uint16_t* base = static_cast<uint16_t*>(out) + idx;
      if constexpr (N == 8) {
        *reinterpret_cast<uint4*>(base) = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                                     pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
      } else {
        *reinterpret_cast<uint2*>(base) = make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
      }
    }
  }
}

// Loads 16 bytes of T (8 bf16 or 4 fp32) as fp32.
template <typename T>
struct Vec16;

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  __device__ __forceinline__ static void load(const void* base, int64_t idx, float (&v)[8]) {
    uint4 u = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx));
    v[0] = bf16_lo(u.x); v[1] = bf16_hi(u.x); v[2] = bf16_lo(u.y); v[3] = bf16_hi(u.y);
    v[4] = bf16_lo(u.z); v[5] = bf16_hi(u.z); v[6] = bf16_lo(u.w); v[7] = bf16_hi(u.w);
  }
  // Unpacks with volatile moves so that the compiler re-expands a packed row on every pass
  // instead of keeping all of its fp32 copies live (which would double the registers).
  __device__ __forceinline__ static void unpack(const uint4& u, float (&v)[8]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      asm volatile("shl.b32 %0, %1, 16;" : "=f"(v[2 * i]) : "r"(w[i]));
      asm volatile("and.b32 %0, %1, 0xFFFF0000;" : "=f"(v[2 * i + 1]) : "r"(w[i]));
    }
  }
};

// 16-byte read-only global load kept in program order with the other volatile asm (so a loop
// of these cannot all be hoisted ahead of the work that consumes them).
__device__ __forceinline__ uint4 ldg16_ordered(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <>
struct Vec16<float> {
  static constexpr int N = 4;
  __device__ __forceinline__ static void load(const void* base, int64_t idx, float (&v)[4]) {
    float4 u = __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx));
    v[0] = u.x; v[1] = u.y; v[2] = u.z; v[3] = u.w;
  }
  __device__ __forceinline__ static void unpack(const uint4& u, float (&v)[4]) {
    asm volatile("mov.b32 %0, %1;" : "=f"(v[0]) : "r"(u.x));
    asm volatile("mov.b32 %0, %1;" : "=f"(v[1]) : "r"(u.y));
    asm volatile("mov.b32 %0, %1;" : "=f"(v[2]) : "r"(u.z));
    asm volatile("mov.b32 %0, %1;" : "=f"(v[3]) : "r"(u.w));
  }
};

// A 16-byte vector of T as packed fp32 pairs (4 pairs of bf16, 2 pairs of fp32).  get() expands
// bf16 with volatile moves, so that a packed row held in registers is re-expanded on each pass
// instead of being kept expanded; cvt() is the plain expansion, free to be scheduled, for data
// that is read from memory right before use.
template <typename T>
struct Pairs;

template <>
struct Pairs<__nv_bfloat16> {
  static constexpr int P = 4;
  __device__ __forceinline__ static void get(const uint4& u, f32x2 (&p)[4]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float lo, hi;
      asm volatile("shl.b32 %0, %1, 16;" : "=f"(lo) : "r"(w[i]));
      asm volatile("and.b32 %0, %1, 0xFFFF0000;" : "=f"(hi) : "r"(w[i]));
      p[i] = f2(lo, hi);
    }
  }
  __device__ __forceinline__ static void cvt(const uint4& u, f32x2 (&p)[4]) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) p[i] = f2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
  }
};

template <>
struct Pairs<float> {
  static constexpr int P = 2;
  __device__ __forceinline__ static void get(const uint4& u, f32x2 (&p)[2]) {
    p[0] = f2(__uint_as_float(u.x), __uint_as_float(u.y));
    p[1] = f2(__uint_as_float(u.z), __uint_as_float(u.w));
  }
  __device__ __forceinline__ static void cvt(const uint4& u, f32x2 (&p)[2]) { get(u, p); }
};

}  // namespace te
