// Row normalization kernels (LayerNorm / RMSNorm forward and backward).
//
// Forward (TransformerEngine JAX "LayerNorm MLP" page, Description step (1); "LayerNorm Dense"
// page, Description): rows of 4, 8 or 16 16-byte vectors per lane of a warp (H = 1024, 2048 or
// 4096 in bf16) take one row per warp, whose sums meet by shuffles alone, each warp loading its
// next row while it works on the current one; bf16 rows of 8192 are shared by the 8 warps of
// one CTA per SM, staged in a 12-row bulk-copy ring; other widths take a CTA of a few warps per
// row, persistent over rows with a stride of the grid, eight CTAs per SM, each thread loading
// the next row's vectors while it normalizes the current one, the warps' row sums meeting in
// shared memory at one barrier per row.  Every form requests its first row before it builds
// its table of gains.  Statistics are fp32, and the normalized row is written once, directly in
// the consumer GEMM's operand dtype (fp32, bf16 or E4M3), together with the per-tensor amax.
//
// Backward (the norm's share of the backward pass, whose gradients cover every parameter):
// rows of x and dz stream through a ring of shared-memory slots, filled by bulk copies (the
// TMA engine's contiguous form) as far ahead as the ring allows, while the CTA's warps work on
// rows already in shared memory.  Each slot has a "full" mbarrier (completed by the copies'
// byte count) and an "empty" one (completed by the warps that read it), and every wait on them
// is bounded; there is no producer warp: the last warp to release a slot issues its refill.
// The row is split across the warps of a CTA (one CTA of 8 warps per SM, or two of 4 for rows
// up to 8 KB); the partial row sums of a few rows at a time meet in shared memory at one named
// barrier.  dgamma and dbeta accumulate per thread in registers, are
// written as one partial row per CTA and summed in a fixed order by a second kernel, so the
// result does not depend on timing.
#include <cstdlib>

#include "cast.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace te {

namespace {

constexpr size_t kRingSmemMax = 224 * 1024;  // dynamic shared memory per CTA
constexpr int kFwdGroupWarps = 4;            // forward: warps per CTA (one row at a time)
constexpr int kFwdRowsCtasPerSm = 8;         // forward: register budget, CTAs per SM
constexpr int kBwdWarps = 8;                 // backward: warps per SM, in one or two CTAs
constexpr int kBwdRowsPerSync = 4;           // backward: rows per barrier (at most)
constexpr int kBwdMaxSlots = 16;

// Barrier `id` among the `nthreads` threads of one group of consumer warps, returning whether
// `pred` was true in any of them.
__device__ __forceinline__ bool group_sync_or(bool pred, int id, int nthreads) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Bytes at the start of the dynamic shared memory: full / empty barriers, the abort flag.
__host__ __device__ constexpr size_t ring_header_bytes(int slots) {
  return (size_t(slots) * 16 + 16 + 127) / 128 * 128;
}

// The CTA's rows are blockIdx.x, blockIdx.x + gridDim.x, ...: its local rows 0 .. nloc - 1.
__device__ __forceinline__ int64_t local_rows(int64_t M) {
  const int64_t b = blockIdx.x, g = gridDim.x;
  return M > b ? (M - b + g - 1) / g : 0;
}

__device__ __forceinline__ void ring_init(uint64_t* full, uint64_t* empty, int slots,
                                          uint32_t empty_count, volatile int* abort_flag) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < slots; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), empty_count);
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
}

// Copies local row k of src0 and the same row of src1 (one behind the other) into slot s,
// completing on the slot's full barrier.
__device__ __forceinline__ void ring_issue(const char* src0, const char* src1, uint32_t row_bytes,
                                           int64_t k, int s, uint8_t* ring, uint64_t* full) {
  const int64_t off = (int64_t(blockIdx.x) + k * gridDim.x) * row_bytes;
  const uint32_t dst = smem_u32(ring + size_t(s) * 2 * row_bytes);
  mbar_expect_tx(smem_u32(&full[s]), 2 * row_bytes);
  bulk_load(dst, src0 + off, row_bytes, smem_u32(&full[s]));
  bulk_load(dst + row_bytes, src1 + off, row_bytes, smem_u32(&full[s]));
}

// A consumer warp's wait for use `use` of slot s: lane 0 waits (bounded) and the warp barrier
// orders the other lanes' reads of the slot after its observation of the completed copy.
// A parity wait tells the awaited phase only from the one before it, so a caller may wait
// for use u only once the slot's use u - 1 has completed (every caller below waits for a slot
// after it has itself consumed the slot's previous use).
__device__ __forceinline__ bool ring_acquire(uint64_t* full, int s, uint32_t use,
                                             volatile int* abort_flag, int* status) {
  const int lane = threadIdx.x & 31;
  int ok = 1;
  if (lane == 0 && !mbar_try_wait(smem_u32(&full[s]), use & 1u))
    ok = wait_bounded(smem_u32(&full[s]), use & 1u, abort_flag, status, kWaitLimitNs, true) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  __syncwarp();
  return ok != 0;
}

// ----------------------------------------------------------------------- forward ---------

// The forward's gain (gamma, plus one when zero-centered) and beta tables in shared memory, as
// fp32: elements 4q .. 4q + 3 of the row's 16-byte vector v sit in float4 q * nvec + v, so a
// lane that owns vector v reads its gains as Q float4s, each warp's reads contiguous.  Filled
// with 16-byte loads of gamma and beta (both 16-byte aligned, the row a whole number of
// vectors) by the CTA's NT threads; with the row's vector count NVEC known at compile time (a
// multiple of NT), every thread's loads are issued back to back.
template <typename T, bool LN, int NT, int NVEC = 0>
__device__ __forceinline__ void fill_gain_table(float4* gain4, float4* beta4, int nvec,
                                                const NormFwdArgs& a, int tid) {
  static_assert(NVEC % NT == 0, "a compile-time row length is a whole number of passes");
  using PR = Pairs<T>;
  constexpr int P = PR::P;
  constexpr int Q = Vec16<T>::N / 4;
  const float shift = a.zero_centered_gamma ? 1.0f : 0.0f;
  const uint4* g = static_cast<const uint4*>(a.gamma);
  const uint4* b = static_cast<const uint4*>(a.beta);
  auto one = [&](int v) {
    f32x2 gp[P], bp[P];
    PR::cvt(__ldg(g + v), gp);
    if (LN && b) PR::cvt(__ldg(b + v), bp);
#pragma unroll
    for (int q = 0; q < Q; ++q) {
      gain4[q * nvec + v] = make_float4(f2lo(gp[2 * q]) + shift, f2hi(gp[2 * q]) + shift,
                                        f2lo(gp[2 * q + 1]) + shift, f2hi(gp[2 * q + 1]) + shift);
      if (LN)
        beta4[q * nvec + v] = b ? make_float4(f2lo(bp[2 * q]), f2hi(bp[2 * q]),
                                              f2lo(bp[2 * q + 1]), f2hi(bp[2 * q + 1]))
                                : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
  };
  if constexpr (NVEC > 0) {
#pragma unroll
    for (int i = 0; i < NVEC / NT; ++i) one(tid + i * NT);
  } else {
    for (int v = tid; v < nvec; v += NT) one(v);
  }
}

// Forward without the ring: one row per CTA of kFwdGroupWarps warps at a time, persistent over
// rows with a stride of the grid.  Each thread loads its NVL 16-byte vectors of the row straight
// into registers, and loads the next row's while it normalizes the current one; many CTAs per
// SM keep enough rows in flight.  The gain and beta sit in shared memory as fp32 float4 blocks
// (fill_gain_table's layout); the warps' row sums meet in shared memory at one barrier per row.
template <typename T, bool LN, int NVL, bool FULL>
__global__ void __launch_bounds__(kFwdGroupWarps * 32, NVL >= 8 ? kFwdRowsCtasPerSm / 2 : kFwdRowsCtasPerSm)
    norm_fwd_rows_kernel(NormFwdArgs a) {
  // the kernel after this one may launch its setup now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using PR = Pairs<T>;
  constexpr int E = Vec16<T>::N;
  constexpr int P = PR::P;
  constexpr int Q = E / 4;
  constexpr int G = kFwdGroupWarps;
  constexpr int GT = G * 32;
  extern __shared__ __align__(16) float4 prm[];
  __shared__ float2 red[2][G];
  const int nvec = int(a.H / E);
  float4* gain4 = prm;
  float4* beta4 = prm + Q * nvec;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto mine = [&](int v) { return FULL || v < nvec; };
  const T* x = static_cast<const T*>(a.x);
  const int64_t stride = gridDim.x;
  auto load_row = [&](int64_t row, uint4 (&r)[NVL], float& first) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + row * a.H) + tid;
#pragma unroll
    for (int i = 0; i < NVL; ++i)
      r[i] = mine(tid + GT * i) ? __ldg(xr + GT * i) : make_uint4(0u, 0u, 0u, 0u);
    if (LN) first = float(x[row * a.H]);
  };
  uint4 bufa[NVL], bufb[NVL];
  float x0a = 0.0f, x0b = 0.0f;
  int64_t row = blockIdx.x;
  // the first row is requested before the gain table is built, so that the table's loads
  // overlap the row's
  if (row < a.M) load_row(row, bufa, x0a);
  fill_gain_table<T, LN, GT>(gain4, beta4, nvec, a, tid);
  __syncthreads();  // gain / beta ready
  const CastState cs = cast_begin(a.cast);
  const float inv_h = 1.0f / float(a.H);
  const bool want_amax = a.cast.amax_out != nullptr;
  float am[P];
#pragma unroll
  for (int p = 0; p < P; ++p) am[p] = 0.0f;
  with_out_amax(out_kind(cs), want_amax, [&](auto tag, auto atag) {
    constexpr int OUT = decltype(tag)::value;
    constexpr bool AMAX = decltype(atag)::value;
    // normalizes row `r` held in `cur` (its first element x0); `par` picks the reduction buffer
    auto process = [&](int64_t r, const uint4 (&cur)[NVL], float x0, int par) {
      f32x2 s1[P], s2[P];
#pragma unroll
      for (int p = 0; p < P; ++p) { s1[p] = f2s(0.0f); s2[p] = f2s(0.0f); }
      const f32x2 x02 = f2s(x0);
#pragma unroll
      for (int i = 0; i < NVL; ++i) {
        if (mine(tid + GT * i)) {
          f32x2 xp[P];
          PR::cvt(cur[i], xp);
#pragma unroll
          for (int p = 0; p < P; ++p) {
            if (LN) {
              const f32x2 d = sub2(xp[p], x02);
              s1[p] = add2(s1[p], d);
              s2[p] = fma2(d, d, s2[p]);
            } else {
              s2[p] = fma2(xp[p], xp[p], s2[p]);
            }
          }
        }
      }
#pragma unroll
      for (int p = 1; p < P; ++p) { s1[0] = add2(s1[0], s1[p]); s2[0] = add2(s2[0], s2[p]); }
      float t1 = LN ? f2lo(s1[0]) + f2hi(s1[0]) : 0.0f;
      float t2 = f2lo(s2[0]) + f2hi(s2[0]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (LN) t1 += __shfl_xor_sync(0xffffffffu, t1, o);
        t2 += __shfl_xor_sync(0xffffffffu, t2, o);
      }
      if (lane == 0) red[par][warp] = make_float2(t1, t2);
      __syncthreads();
      t1 = 0.0f;
      t2 = 0.0f;
#pragma unroll
      for (int w = 0; w < G; ++w) {  // warp order: the same bits in every thread
        const float2 rr = red[par][w];
        t1 += rr.x;
        t2 += rr.y;
      }
      const float m1 = LN ? t1 * inv_h : 0.0f;
      const float m2 = t2 * inv_h;
      const float mean = LN ? x0 + m1 : 0.0f;
      const float var = LN ? fmaxf(m2 - m1 * m1, 0.0f) : m2;
      const float rs = rsqrtf(var + a.eps);
      if (tid == 0) {
        if (a.mu) a.mu[r] = mean;
        if (a.rsigma) a.rsigma[r] = rs;
      }
      if (OUT != OUT_NONE || AMAX) {
        const f32x2 mean2 = f2s(mean), rs2 = f2s(rs);
        const int64_t base = r * a.H + int64_t(tid) * E;
#pragma unroll
        for (int i = 0; i < NVL; ++i) {
          const int v = tid + GT * i;
          if (mine(v)) {
            f32x2 xp[P], gp[P], bp[P];
            PR::cvt(cur[i], xp);
#pragma unroll
            for (int q = 0; q < Q; ++q) {
              const float4 g4 = gain4[q * nvec + v];
              gp[2 * q] = f2(g4.x, g4.y);
              gp[2 * q + 1] = f2(g4.z, g4.w);
              if (LN) {
                const float4 b4 = beta4[q * nvec + v];
                bp[2 * q] = f2(b4.x, b4.y);
                bp[2 * q + 1] = f2(b4.z, b4.w);
              }
            }
            float y[E];
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const f32x2 yy = LN ? fma2(sub2(xp[p], mean2), mul2(gp[p], rs2), bp[p])
                                  : mul2(mul2(xp[p], rs2), gp[p]);
              if (AMAX) am[p] = absmax2(am[p], yy);
              y[2 * p] = f2lo(yy);
              y[2 * p + 1] = f2hi(yy);
            }
            store_out<OUT, E>(a.out, base + int64_t(GT) * E * i, y, cs);
          }
        }
      }
    };
    // two register buffers in turn: the next row loads while the current one is processed;
    // the rows after it are asked into L2 by one thread
    const uint32_t row_bytes = uint32_t(a.H) * uint32_t(sizeof(T));
    auto prefetch_ahead = [&](int64_t r) {
      if (tid == 0 && a.prefetch > 0 && r + (a.prefetch + 1) * stride < a.M)
        bulk_prefetch_l2(x + (r + (a.prefetch + 1) * stride) * a.H, row_bytes);
    };
    if (tid == 0)
      for (int k = 2; k <= a.prefetch && row + k * stride < a.M; ++k)
        bulk_prefetch_l2(x + (row + k * stride) * a.H, row_bytes);
    for (int par = 0; row < a.M; par ^= 1) {
      prefetch_ahead(row);
      if (row + stride < a.M) load_row(row + stride, bufb, x0b);
      process(row, bufa, x0a, par);
      row += stride;
      par ^= 1;
      if (row >= a.M) break;
      prefetch_ahead(row);
      if (row + stride < a.M) load_row(row + stride, bufa, x0a);
      process(row, bufb, x0b, par);
      row += stride;
    }
  });
  float amax = am[0];
#pragma unroll
  for (int p = 1; p < P; ++p) amax = fmaxf(amax, am[p]);
  amax = warp_max(amax);
  if (lane == 0 && a.cast.amax_out) atomic_max_nonneg(a.cast.amax_out, amax);
}

// Forward with one row per warp, for rows of exactly NVW x 32 vectors: the row's sums meet by
// shuffles within the warp, with no barrier between warps; the CTA's kFwdWarpRowWarps warps
// share the gain / beta table in shared memory (fill_gain_table's layout).  Each lane holds its
// NVW vectors of one row (PIPE: of two rows, the next one loading while the current one is
// worked on); the many warps per SM keep rows in flight.  The output kind and the amax are
// template parameters, picked on the host: one kernel holds one fully unrolled row loop
// (measured against one kernel holding every kind's loop: E4M3 output +3% at 8192 x 4096, +2%
// LayerNorm at 16384 x 4096, with fewer registers).
constexpr int kFwdWarpRowWarps = 4;
__host__ __device__ constexpr int fwd_warp_ctas(int elems_per_lane, bool pipe) {
  return pipe ? (elems_per_lane >= 128 ? 2 : 3) : (elems_per_lane >= 128 ? 3 : 4);
}
template <typename T, bool LN, int NVW, bool PIPE, int OUT, bool AMAX>
__global__ void __launch_bounds__(kFwdWarpRowWarps * 32, fwd_warp_ctas(NVW * Vec16<T>::N, PIPE))
    norm_fwd_warp_kernel(NormFwdArgs a) {
  // the kernel after this one may launch its setup now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using PR = Pairs<T>;
  constexpr int E = Vec16<T>::N;
  constexpr int P = PR::P;
  constexpr int Q = E / 4;
  constexpr int nvec = NVW * 32;
  extern __shared__ __align__(16) float4 prm[];
  float4* gain4 = prm;
  float4* beta4 = prm + Q * nvec;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const T* x = static_cast<const T*>(a.x);
  const int64_t step = int64_t(gridDim.x) * kFwdWarpRowWarps;
  const int64_t r_first = int64_t(blockIdx.x) * kFwdWarpRowWarps + warp;
  // PIPE: the warp's first row is requested before the gain table is built, so that the
  // table's loads overlap the row's
  uint4 cur[NVW];
  if (PIPE && r_first < a.M) {
    const uint4* xr = reinterpret_cast<const uint4*>(x + r_first * a.H) + lane;
#pragma unroll
    for (int i = 0; i < NVW; ++i) cur[i] = __ldg(xr + 32 * i);
  }
  fill_gain_table<T, LN, kFwdWarpRowWarps * 32, nvec>(gain4, beta4, nvec, a, tid);
  __syncthreads();  // gain / beta ready
  const CastState cs = cast_begin(a.cast);
  const float inv_h = 1.0f / float(a.H);
  float am[P];
#pragma unroll
  for (int p = 0; p < P; ++p) am[p] = 0.0f;
  {
    for (int64_t r = r_first; r < a.M; r += step) {
      // PIPE: the warp's next row is requested before this row's arithmetic, so that a row's
      // loads are always in flight
      uint4 nxt[NVW];
      if (PIPE) {
        if (r + step < a.M) {
          const uint4* xn = reinterpret_cast<const uint4*>(x + (r + step) * a.H) + lane;
#pragma unroll
          for (int i = 0; i < NVW; ++i) nxt[i] = __ldg(xn + 32 * i);
        }
      } else {
        const uint4* xr = reinterpret_cast<const uint4*>(x + r * a.H) + lane;
#pragma unroll
        for (int i = 0; i < NVW; ++i) cur[i] = __ldg(xr + 32 * i);
      }
      // the row's first element, subtracted before the sums (shifted variance), from lane 0
      float x0 = 0.0f;
      if (LN) {
        f32x2 first[P];
        PR::cvt(cur[0], first);
        x0 = __shfl_sync(0xffffffffu, f2lo(first[0]), 0);
      }
      const f32x2 x02 = f2s(x0);
      f32x2 s1[P], s2[P];
#pragma unroll
      for (int p = 0; p < P; ++p) { s1[p] = f2s(0.0f); s2[p] = f2s(0.0f); }
#pragma unroll
      for (int i = 0; i < NVW; ++i) {
        f32x2 xp[P];
        PR::cvt(cur[i], xp);
#pragma unroll
        for (int p = 0; p < P; ++p) {
          if (LN) {
            const f32x2 d = sub2(xp[p], x02);
            s1[p] = add2(s1[p], d);
            s2[p] = fma2(d, d, s2[p]);
          } else {
            s2[p] = fma2(xp[p], xp[p], s2[p]);
          }
        }
      }
#pragma unroll
      for (int p = 1; p < P; ++p) { s1[0] = add2(s1[0], s1[p]); s2[0] = add2(s2[0], s2[p]); }
      float t1 = LN ? f2lo(s1[0]) + f2hi(s1[0]) : 0.0f;
      float t2 = f2lo(s2[0]) + f2hi(s2[0]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        if (LN) t1 += __shfl_xor_sync(0xffffffffu, t1, o);
        t2 += __shfl_xor_sync(0xffffffffu, t2, o);
      }
      const float m1 = LN ? t1 * inv_h : 0.0f;
      const float m2 = t2 * inv_h;
      const float mean = LN ? x0 + m1 : 0.0f;
      const float var = LN ? fmaxf(m2 - m1 * m1, 0.0f) : m2;
      const float rs = rsqrtf(var + a.eps);
      if (lane == 0) {
        if (a.mu) a.mu[r] = mean;
        if (a.rsigma) a.rsigma[r] = rs;
      }
      if (OUT != OUT_NONE || AMAX) {
        const f32x2 mean2 = f2s(mean), rs2 = f2s(rs);
        const int64_t base = r * a.H + int64_t(lane) * E;
#pragma unroll
        for (int i = 0; i < NVW; ++i) {
          const int v = lane + 32 * i;
          f32x2 xp[P], gp[P], bp[P];
          PR::get(cur[i], xp);  // converted again here rather than kept from the sums
#pragma unroll
          for (int q = 0; q < Q; ++q) {
            const float4 g4 = gain4[q * nvec + v];
            gp[2 * q] = f2(g4.x, g4.y);
            gp[2 * q + 1] = f2(g4.z, g4.w);
            if (LN) {
              const float4 b4 = beta4[q * nvec + v];
              bp[2 * q] = f2(b4.x, b4.y);
              bp[2 * q + 1] = f2(b4.z, b4.w);
            }
          }
          float y[E];
#pragma unroll
          for (int p = 0; p < P; ++p) {
            const f32x2 yy = LN ? fma2(sub2(xp[p], mean2), mul2(gp[p], rs2), bp[p])
                                : mul2(mul2(xp[p], rs2), gp[p]);
            if (AMAX) am[p] = absmax2(am[p], yy);
            y[2 * p] = f2lo(yy);
            y[2 * p + 1] = f2hi(yy);
          }
          store_out<OUT, E>(a.out, base + int64_t(32) * E * i, y, cs);
          // one vector's gain / beta loads at a time: hoisting all of them spills
          asm volatile("" ::: "memory");
        }
      }
      if (PIPE) {
#pragma unroll
        for (int i = 0; i < NVW; ++i) cur[i] = nxt[i];
      }
    }
  }
  float amax = am[0];
#pragma unroll
  for (int p = 1; p < P; ++p) amax = fmaxf(amax, am[p]);
  amax = warp_max(amax);
  if (lane == 0 && a.cast.amax_out) atomic_max_nonneg(a.cast.amax_out, amax);
}

// Sets the kernel's dynamic shared memory limit once per device; `max_carveout` also asks for
// the largest shared-memory share of the SM's L1 (for two large-ring CTAs per SM; the forward
// kernels, which read through L1, measured slower with it).
template <typename K>
te_status allow_ring_smem(K kernel, PerDevice<bool>& done, bool max_carveout = false) {
  bool ok = false;
  return done.get(&ok, [&](bool* v) {
           *v = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     int(kRingSmemMax)) == cudaSuccess &&
                (!max_carveout ||
                 cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                      int(cudaSharedmemCarveoutMaxShared)) == cudaSuccess);
           return *v;
         })
             ? TE_OK
             : TE_ERR_CUDA;
}

// Ring size for `slot_bytes`-byte slots: as many as fit the shared memory (at most
// max_slots), rounded down to a multiple of `mult`; 0 if fewer than `min_slots` fit.
int ring_slots(size_t slot_bytes, int max_slots, int min_slots, int mult,
               size_t max_bytes = kRingSmemMax) {
  int slots = max_slots;
  while (slots > 0 && ring_header_bytes(slots) + size_t(slots) * slot_bytes > max_bytes)
    --slots;
  slots -= slots % mult;
  return slots >= min_slots ? slots : 0;
}

// Rows ahead of its current row that a warp (or a row group) of the forward asks L2 to fetch:
// `fallback` unless TE_NORM_FWD_PREFETCH (0 .. 8) in the environment says otherwise (a switch
// for measurements).  The row-group kernel gains from one row ahead (its next row is already
// loading into registers); the one-row-per-warp kernel measured no gain.
int fwd_prefetch_rows(int fallback) {
  static const int env = [] {
    const char* e = getenv("TE_NORM_FWD_PREFETCH");
    if (!e) return -1;
    const int v = atoi(e);
    return v < 0 ? 0 : v > 8 ? 8 : v;
  }();
  return env >= 0 ? env : fallback;
}

template <typename T, bool LN, int NVL, bool FULL>
te_status launch_fwd_rows(const NormFwdArgs& a_in, cudaStream_t s) {
  NormFwdArgs a = a_in;
  a.prefetch = fwd_prefetch_rows(1);
  static PerDevice<bool> attr_done;
  const size_t params = size_t(a.H) * (LN ? 2 : 1) * sizeof(float);
  const te_status st = allow_ring_smem(norm_fwd_rows_kernel<T, LN, NVL, FULL>, attr_done);
  if (st != TE_OK) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, norm_fwd_rows_kernel<T, LN, NVL, FULL>,
                                                    kFwdGroupWarps * 32, params) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t cap = int64_t(num_sms()) * per_sm;
  const unsigned grid = unsigned(a.M < cap ? a.M : cap);
  norm_fwd_rows_kernel<T, LN, NVL, FULL><<<grid, kFwdGroupWarps * 32, params, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T, bool LN, int NVW, bool PIPE, int OUT, bool AMAX>
te_status launch_fwd_warp_kind(const NormFwdArgs& a, cudaStream_t s) {
  static PerDevice<bool> attr_done;
  auto* kernel = norm_fwd_warp_kernel<T, LN, NVW, PIPE, OUT, AMAX>;
  const size_t params = size_t(a.H) * (LN ? 2 : 1) * sizeof(float);
  const te_status st = allow_ring_smem(kernel, attr_done);
  if (st != TE_OK) return st;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kFwdWarpRowWarps * 32,
                                                    params) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int64_t cap = int64_t(num_sms()) * per_sm;
  const int64_t ctas = ceil_div(a.M, kFwdWarpRowWarps);
  const unsigned grid = unsigned(ctas < cap ? ctas : cap);
  kernel<<<grid, kFwdWarpRowWarps * 32, params, s>>>(a);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T, bool LN, int NVW, bool PIPE>
te_status launch_fwd_warp(const NormFwdArgs& a, cudaStream_t s) {
  te_status st = TE_ERR_UNSUPPORTED;
  with_out_amax(out_kind_of(a.cast.store, a.cast.out_dtype, a.cast.fake_quant),
                a.cast.amax_out != nullptr, [&](auto tag, auto atag) {
                  st = launch_fwd_warp_kind<T, LN, NVW, PIPE, decltype(tag)::value,
                                            decltype(atag)::value>(a, s);
                });
  return st;
}

// Forward for long rows (exactly kFwdCtaWarps x 32 x NV 16-byte vectors: H = 8192 bf16 with
// NV = 4): the 8 warps of one CTA per SM share each row, as in the backward.  The
// CTA's rows (blockIdx.x, blockIdx.x + gridDim.x, ...) arrive by cp.async.bulk in a ring of
// `spc` shared-memory slots of one row each (12 at 16 KB), so that up to 12 rows per SM are in
// flight without occupying registers.  The CTA works on RB rows at a time: each thread takes
// its NV vectors of each of them into registers and releases their slots; its gain and beta
// vectors stay in registers for the whole kernel.  The warps' partial sums of the RB rows meet
// at one named barrier (double-buffered, and carrying a failed wait so that the warps stop
// together); after it one warp per row, in turn, waits for the slot's release and refills it
// with the row `spc` ahead.  Every wait is bounded.
constexpr int kFwdCtaWarps = 8;
constexpr int kFwdCtaVecs = 1024 / (kFwdCtaWarps * 32);  // vectors per thread per row
constexpr int kFwdCtaMaxSlots = 16;
// Rows per barrier: 2, and 4 with E4M3 output, whose longer chain of dependent arithmetic per
// row gains from the wider step (measured at 16384 x 8192: bf16 output 7% slower with 4 rows,
// E4M3 output 2% faster; 1 row slower for both; 16 warps slower; for 4096-wide rows two CTAs of
// 4 warps per SM measured 10-30% slower than one row per warp).
constexpr int kFwdCtaRows = 2;
constexpr int kFwdCtaRowsE4M3 = 4;

template <typename T, bool LN, int NV, int G, int RB>
__global__ void __launch_bounds__(G * 32, G < 8 ? 8 / G : 1)
    norm_fwd_cta_kernel(NormFwdArgs a, int* status, int spc) {
  // the kernel after this one may launch its setup now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  using PR = Pairs<T>;
  constexpr int E = Vec16<T>::N;
  constexpr int P = PR::P;
  constexpr int GT = G * 32;
  constexpr uint32_t row_bytes = uint32_t(GT * NV) * 16u;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float2 red[2][RB][G];
  __shared__ int last_use[kFwdCtaMaxSlots];  // the latest use issued into each slot
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + spc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + spc);
  uint8_t* ring = smem + ring_header_bytes(spc);
  const char* xb = static_cast<const char*>(a.x);
  const int64_t nloc = local_rows(a.M);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // local row k -> slot sl: its copy completes on full[sl]
  auto issue = [&](int64_t k, int sl) {
    const int64_t row = int64_t(blockIdx.x) + k * gridDim.x;
    mbar_expect_tx(smem_u32(&full[sl]), row_bytes);
    bulk_load(smem_u32(ring + size_t(sl) * row_bytes), xb + row * row_bytes, row_bytes,
              smem_u32(&full[sl]));
  };
  if (tid < spc) last_use[tid] = -1;
  ring_init(full, empty, spc, G, abort_flag);
  if (tid == 0) {  // the first use of every slot (the barriers' init is fenced)
    for (int k = 0; k < spc && k < nloc; ++k) {
      issue(k, k);
      last_use[k] = 0;
    }
  }
  // this thread's gain (and beta) vectors, as fp32 pairs, while the first rows load
  f32x2 gp[NV][P], bp[NV][P];
  {
    const f32x2 shift = f2s(a.zero_centered_gamma ? 1.0f : 0.0f);
#pragma unroll
    for (int i = 0; i < NV; ++i) {
      const int v = tid + i * GT;
      PR::cvt(__ldg(reinterpret_cast<const uint4*>(a.gamma) + v), gp[i]);
      if (LN && a.beta) PR::cvt(__ldg(reinterpret_cast<const uint4*>(a.beta) + v), bp[i]);
#pragma unroll
      for (int p = 0; p < P; ++p) {
        gp[i][p] = add2(gp[i][p], shift);
        if (!LN || !a.beta) bp[i][p] = f2s(0.0f);
      }
    }
  }
  const CastState cs = cast_begin(a.cast);
  const float inv_h = 1.0f / float(a.H);
  const bool want_amax = a.cast.amax_out != nullptr;
  float am[P];
#pragma unroll
  for (int p = 0; p < P; ++p) am[p] = 0.0f;
  with_out_amax(out_kind(cs), want_amax, [&](auto tag, auto atag) {
    constexpr int OUT = decltype(tag)::value;
    constexpr bool AMAX = decltype(atag)::value;
    int s0 = 0;  // the step's rows are in slots s0 .. s0 + nr - 1 (spc is a multiple of RB)
    uint32_t use = 0;
    for (int64_t j0 = 0, it = 0; j0 < nloc; j0 += RB, ++it) {
      const int nr = nloc - j0 < RB ? int(nloc - j0) : RB;
      bool ok = true;
#pragma unroll
      for (int r = 0; r < RB; ++r)
        if (r < nr && ok) ok = ring_acquire(full, s0 + r, use, abort_flag, status);
      uint4 cur[RB][NV];
      float x0[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        x0[r] = 0.0f;
#pragma unroll
        for (int i = 0; i < NV; ++i) cur[r][i] = make_uint4(0u, 0u, 0u, 0u);
        if (ok && r < nr) {
          const uint4* src = reinterpret_cast<const uint4*>(ring + size_t(s0 + r) * row_bytes);
#pragma unroll
          for (int i = 0; i < NV; ++i) cur[r][i] = src[tid + i * GT];
          if (LN) {  // the row's first element, subtracted before the sums (shifted variance)
            f32x2 first[P];
            PR::cvt(src[0], first);
            x0[r] = f2lo(first[0]);
          }
        }
      }
      // the rows are in registers: their slots may be refilled
      __syncwarp();
      if (lane == 0 && ok) {
#pragma unroll
        for (int r = 0; r < RB; ++r)
          if (r < nr) mbar_arrive(smem_u32(&empty[s0 + r]));
      }
      float t1[RB], t2[RB];
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const f32x2 x02 = f2s(x0[r]);
        f32x2 s1[P], s2[P];
#pragma unroll
        for (int p = 0; p < P; ++p) { s1[p] = f2s(0.0f); s2[p] = f2s(0.0f); }
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          f32x2 xp[P];
          PR::cvt(cur[r][i], xp);
#pragma unroll
          for (int p = 0; p < P; ++p) {
            if (LN) {
              const f32x2 d = sub2(xp[p], x02);
              s1[p] = add2(s1[p], d);
              s2[p] = fma2(d, d, s2[p]);
            } else {
              s2[p] = fma2(xp[p], xp[p], s2[p]);
            }
          }
        }
#pragma unroll
        for (int p = 1; p < P; ++p) { s1[0] = add2(s1[0], s1[p]); s2[0] = add2(s2[0], s2[p]); }
        t1[r] = LN ? f2lo(s1[0]) + f2hi(s1[0]) : 0.0f;
        t2[r] = f2lo(s2[0]) + f2hi(s2[0]);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          if (LN) t1[r] += __shfl_xor_sync(0xffffffffu, t1[r], o);
          t2[r] += __shfl_xor_sync(0xffffffffu, t2[r], o);
        }
      }
      const int par = int(it & 1);
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) red[par][r][warp] = make_float2(t1[r], t2[r]);
      }
      if (group_sync_or(!ok, 1, GT)) break;
      // every warp has released the step's slots: one warp per slot, in turn, refills it with
      // the row spc ahead (its wait on the slot's empty barrier acquires the other warps' reads)
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int sl = s0 + r;
        if (warp == int((j0 + r) % G) && lane == 0 && r < nr && j0 + r + spc < nloc &&
            (mbar_try_wait(smem_u32(&empty[sl]), use & 1u) ||
             wait_bounded(smem_u32(&empty[sl]), use & 1u, abort_flag, status, kWaitLimitNs, true))) {
          fence_proxy_async_smem();
          issue(j0 + r + spc, sl);
          last_use[sl] = int(use) + 1;
        }
      }
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        if (r >= nr) break;
        // the warps' sums in warp order (the same bits in every thread)
        float r1 = 0.0f, r2 = 0.0f;
#pragma unroll
        for (int w = 0; w < G; ++w) {
          const float2 v = red[par][r][w];
          r1 += v.x;
          r2 += v.y;
        }
        const int64_t row = int64_t(blockIdx.x) + (j0 + r) * gridDim.x;
        const float m1 = LN ? r1 * inv_h : 0.0f;
        const float m2 = r2 * inv_h;
        const float mean = LN ? x0[r] + m1 : 0.0f;
        const float var = LN ? fmaxf(m2 - m1 * m1, 0.0f) : m2;
        const float rs = rsqrtf(var + a.eps);
        if (tid == 0) {
          if (a.mu) a.mu[row] = mean;
          if (a.rsigma) a.rsigma[row] = rs;
        }
        if (OUT != OUT_NONE || AMAX) {
          const f32x2 mean2 = f2s(mean), rs2 = f2s(rs);
#pragma unroll
          for (int i = 0; i < NV; ++i) {
            f32x2 xp[P];
            PR::get(cur[r][i], xp);
            float y[E];
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const f32x2 yy = LN ? fma2(sub2(xp[p], mean2), mul2(gp[i][p], rs2), bp[i][p])
                                  : mul2(mul2(xp[p], rs2), gp[i][p]);
              if (AMAX) am[p] = absmax2(am[p], yy);
              y[2 * p] = f2lo(yy);
              y[2 * p + 1] = f2hi(yy);
            }
            store_out<OUT, E>(a.out, row * a.H + int64_t(tid + i * GT) * E, y, cs);
          }
        }
      }
      s0 += RB;
      if (s0 == spc) {
        s0 = 0;
        ++use;
      }
    }
  });
  // After a failed wait, copies issued but never consumed may still be in flight: wait for them
  // (briefly) before the CTA exits.  Without a failure every issued row was consumed.
  __syncthreads();
  if (tid == 0 && *abort_flag) {
    for (int k = 0; k < spc; ++k)
      if (last_use[k] >= 0)
        wait_bounded(smem_u32(&full[k]), uint32_t(last_use[k]) & 1u, nullptr, status,
                     kDrainLimitNs, false);
  }
  float amax = am[0];
#pragma unroll
  for (int p = 1; p < P; ++p) amax = fmaxf(amax, am[p]);
  amax = warp_max(amax);
  if (lane == 0 && a.cast.amax_out) atomic_max_nonneg(a.cast.amax_out, amax);
}

template <typename T, bool LN, int NV, int G, int RB>
te_status launch_fwd_cta_rb(const NormFwdArgs& a, cudaStream_t s) {
  static PerDevice<bool> attr_done;
  constexpr size_t row_bytes = size_t(G) * 32 * NV * 16;
  constexpr int kCtas = G < 8 ? 8 / G : 1;  // CTAs per SM, sharing its shared memory
  const size_t cap = kCtas == 1 ? kRingSmemMax : size_t(227 * 1024) / kCtas - 1024;
  // a step holds RB slots; a second step's worth lets the refills run ahead
  const int spc = ring_slots(row_bytes, kFwdCtaMaxSlots, 2 * RB, RB, cap);
  if (spc == 0) return TE_ERR_UNSUPPORTED;
  const te_status st =
      allow_ring_smem(norm_fwd_cta_kernel<T, LN, NV, G, RB>, attr_done, kCtas > 1);
  if (st != TE_OK) return st;
  const size_t smem = ring_header_bytes(spc) + size_t(spc) * row_bytes;
  const int64_t n = int64_t(num_sms()) * kCtas;
  const unsigned grid = unsigned(a.M < n ? a.M : n);
  norm_fwd_cta_kernel<T, LN, NV, G, RB><<<grid, G * 32, smem, s>>>(a, device_status_ptr(), spc);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <typename T, bool LN, int NV, int G>
te_status launch_fwd_cta(const NormFwdArgs& a, cudaStream_t s) {
  return a.cast.out_dtype == TE_E4M3 && a.cast.store
             ? launch_fwd_cta_rb<T, LN, NV, G, kFwdCtaRowsE4M3>(a, s)
             : launch_fwd_cta_rb<T, LN, NV, G, kFwdCtaRows>(a, s);
}

// One row per warp, loaded straight into registers, each warp requesting its next row before
// the current row's arithmetic (with two rows in registers fewer warps fit an SM; measured
// against one row at a time: equal with bf16 output and 1% faster with E4M3 at 8192 x 4096, 3%
// faster at 8192 x 2048).  TE_NORM_FWD_KERNEL=warp in the environment forces the one-row-at-a-
// time form (a switch between complete kernels, for measurements).
template <typename T, int NVW>
te_status launch_fwd_nvw(const NormFwdArgs& a, cudaStream_t s) {
  static const bool one_row = [] {
    const char* e = getenv("TE_NORM_FWD_KERNEL");
    return e && e[0] == 'w';
  }();
  const bool ln = a.norm_type == TE_LAYERNORM;
  if (one_row)
    return ln ? launch_fwd_warp<T, true, NVW, false>(a, s) : launch_fwd_warp<T, false, NVW, false>(a, s);
  return ln ? launch_fwd_warp<T, true, NVW, true>(a, s) : launch_fwd_warp<T, false, NVW, true>(a, s);
}

template <typename T, int NVL>
te_status launch_fwd_nvl(const NormFwdArgs& a, cudaStream_t s) {
  // (the bounds-tested form throughout: without the tests the compiler holds more of the two
  // row buffers live and spills)
  return a.norm_type == TE_LAYERNORM ? launch_fwd_rows<T, true, NVL, false>(a, s)
                                     : launch_fwd_rows<T, false, NVL, false>(a, s);
}

template <typename T>
te_status launch_fwd_t(const NormFwdArgs& a, cudaStream_t s) {
  constexpr int E = Vec16<T>::N;
  constexpr int GT = kFwdGroupWarps * 32;
  // rows are at most 16 KB, i.e. 1024 vectors
  constexpr int kMaxNVL = (1024 + GT - 1) / GT;
  // rows of 4, 8 or 16 vectors per lane of one warp: one row per warp
  const int64_t nvec = a.H / E;
  if (nvec % 32 == 0) {
    if (nvec == 4 * 32) return launch_fwd_nvw<T, 4>(a, s);
    if (nvec == 8 * 32) return launch_fwd_nvw<T, 8>(a, s);
    if (nvec == 16 * 32) return launch_fwd_nvw<T, 16>(a, s);
  }
  // bf16 rows of 1024 vectors (H = 8192): shared by the 8 warps of one CTA per SM, staged in a
  // ring (measured against the register kernel below at 16384 / 8192 rows: bf16 output +15% /
  // +28%, E4M3 output +8% / +19%; fp32 rows of 4096 measured slower that way and stay there).
  // TE_NORM_FWD_LONG=rows in the environment forces the register kernel (a switch between two
  // complete kernels, for measurements).
  static const bool long_rows = [] {
    const char* e = getenv("TE_NORM_FWD_LONG");
    return !(e && e[0] == 'r');
  }();
  if constexpr (sizeof(T) == 2) {
    if (long_rows && nvec == int64_t(kFwdCtaWarps) * 32 * kFwdCtaVecs)
      return a.norm_type == TE_LAYERNORM ? launch_fwd_cta<T, true, kFwdCtaVecs, kFwdCtaWarps>(a, s)
                                         : launch_fwd_cta<T, false, kFwdCtaVecs, kFwdCtaWarps>(a, s);
  }
  const int64_t per_thread = ceil_div(a.H / E, GT);
  if (per_thread <= 1) return launch_fwd_nvl<T, 1>(a, s);
  if (per_thread <= 2) return launch_fwd_nvl<T, 2>(a, s);
  if (per_thread <= 4) return launch_fwd_nvl<T, 4>(a, s);
  if constexpr (kMaxNVL > 4) {
    if (per_thread <= 8) return launch_fwd_nvl<T, 8>(a, s);
  }
  if constexpr (kMaxNVL > 8) {
    if (per_thread <= 16) return launch_fwd_nvl<T, 16>(a, s);
  }
  if constexpr (kMaxNVL > 16) {
    if (per_thread <= 32) return launch_fwd_nvl<T, 32>(a, s);
  }
  return TE_ERR_UNSUPPORTED;
}

// ----------------------------------------------------------------------- backward --------

// All G warps of a CTA share each of its rows: thread t owns the 16-byte vectors t,
// t + 32 * G, ... of the row (NV of them), with its gamma vectors and dgamma / dbeta
// accumulators in registers.  The CTA's rows (local rows 0, 1, ...) go round a ring of `spc`
// slots, each holding one row of x followed by the same row of dz; RB consecutive rows form a
// step, whose row sums meet in shared memory at one named barrier, which also carries each
// warp's "wait failed" flag so that the warps stop together.  There is no producer warp: after
// its first pass over a slot each warp arrives on the slot's empty barrier, and after the
// step's barrier one warp waits for those (which acquires the others' reads) and issues the
// bulk copies of the rows `spc` rows ahead into the slots.  With no ninth warp a thread may
// hold up to 255 registers, enough to keep xhat and dz * g of the step's rows for the second
// pass instead of reading and converting the slot again.
__host__ __device__ constexpr int bwd_rows_per_sync(int nv) { return nv >= 4 ? 1 : kBwdRowsPerSync; }

template <typename T, bool LN, int NV, bool FULL, int G>
__global__ void __launch_bounds__(G * 32, kBwdWarps / G)
    norm_bwd_ring_kernel(NormBwdArgs a, int* status, int spc) {
  using PR = Pairs<T>;
  constexpr int E = Vec16<T>::N;
  constexpr int P = PR::P;
  constexpr int GT = G * 32;
  constexpr int RB = bwd_rows_per_sync(NV);
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ float2 red[2][RB][G];
  __shared__ int last_use[kBwdMaxSlots];  // the latest use issued into each slot
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + spc;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + spc);
  uint8_t* ring = smem + ring_header_bytes(spc);
  const char* xsrc = static_cast<const char*>(a.x);
  const char* dzsrc = static_cast<const char*>(a.dz);
  const int nvec = int(a.H / E);
  const uint32_t row_bytes = uint32_t(a.H) * uint32_t(sizeof(T));
  const uint32_t slot_bytes = 2 * row_bytes;
  const int64_t nloc = local_rows(a.M);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < spc) last_use[threadIdx.x] = -1;
  ring_init(full, empty, spc, G, abort_flag);
  // the column-sum kernel that follows may launch now: it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) {  // the first use of every slot (the barriers' init is fenced)
    for (int k = 0; k < spc && k < nloc; ++k) {
      ring_issue(xsrc, dzsrc, row_bytes, k, k, ring, full);
      last_use[k] = 0;
    }
  }

  // FULL: every thread owns exactly NV vectors of every row (no bounds tests)
  auto mine = [&](int v) { return FULL || v < nvec; };
  const int gt = threadIdx.x;
  const float inv_h = 1.0f / float(a.H);
  const f32x2 gshift = f2s(a.zero_centered_gamma ? 1.0f : 0.0f);
  f32x2 gp[NV][P], accg[NV][P], accb[NV][P];
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = gt + i * GT;
    const uint4 graw = mine(v) ? __ldg(reinterpret_cast<const uint4*>(a.gamma) + v)
                               : make_uint4(0u, 0u, 0u, 0u);
    PR::cvt(graw, gp[i]);
#pragma unroll
    for (int p = 0; p < P; ++p) {
      gp[i][p] = add2(gp[i][p], gshift);
      accg[i][p] = f2s(0.0f);
      accb[i][p] = f2s(0.0f);
    }
  }
  // local row k is global row blockIdx.x + k * gridDim.x
  const int64_t row_step = gridDim.x;
  float mu_n[RB], rs_n[RB];
#pragma unroll
  for (int j = 0; j < RB; ++j) {
    const int64_t row = blockIdx.x + j * row_step;
    mu_n[j] = (LN && j < nloc) ? a.mu[row] : 0.0f;
    rs_n[j] = j < nloc ? a.rsigma[row] : 0.0f;
  }
  const int64_t dx_step = row_step * a.H;
  int jj = 0;
  uint32_t use = 0;
  int64_t row0 = blockIdx.x;
  T* dx0 = static_cast<T*>(a.dx) + row0 * a.H + gt * E;
  bool ok = true;
  for (int64_t j0 = 0, it = 0; j0 < nloc;
       j0 += RB, ++it, row0 += RB * row_step, dx0 += RB * dx_step) {
    const int nr = nloc - j0 < RB ? int(nloc - j0) : RB;
    // xhat = x * rs - mu * rs, one fused multiply-add per pair: mu * rs is rounded once, an
    // error near 2^-24 |mu| rs in xhat, below the bf16 output's resolution unless the row's
    // mean exceeds its standard deviation by some 10^4
    f32x2 nmr2[RB], rs2[RB];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      nmr2[j] = f2s(-mu_n[j] * rs_n[j]);
      rs2[j] = f2s(rs_n[j]);
      if (j0 + RB + j < nloc) {  // the next step's statistics load while this step runs
        const int64_t row = row0 + (RB + j) * row_step;
        mu_n[j] = LN ? a.mu[row] : 0.0f;
        rs_n[j] = a.rsigma[row];
      }
    }
    const int s0 = jj;  // the step's rows are in slots s0 .. s0 + nr - 1 (spc is a multiple of RB)
    const uint8_t* slot0 = ring + uint32_t(s0) * slot_bytes;
#pragma unroll
    for (int j = 0; j < RB; ++j)
      if (j < nr && ok) ok = ring_acquire(full, s0 + j, use, abort_flag, status);
    // pass 1, over the rows in shared memory: the two row sums sum(dz * g) and
    // sum(dz * g * xhat), and the column sums dgamma += dz * xhat, dbeta += dz (which do not
    // depend on the row sums); xhat and dz * g stay in registers for pass 2
    float t1[RB], t2[RB];
    f32x2 xk[RB][NV][P], gk[RB][NV][P];
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      f32x2 s1 = f2s(0.0f), s2 = f2s(0.0f);
#pragma unroll
      for (int i = 0; i < NV; ++i)
#pragma unroll
        for (int p = 0; p < P; ++p) { xk[j][i][p] = f2s(0.0f); gk[j][i][p] = f2s(0.0f); }
      if (ok && j < nr) {
        const uint4* xs = reinterpret_cast<const uint4*>(slot0 + j * slot_bytes) + gt;
        const uint4* dzs = xs + nvec;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          if (mine(gt + i * GT)) {
            f32x2 xp[P], dp[P];
            PR::cvt(xs[i * GT], xp);
            PR::cvt(dzs[i * GT], dp);
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const f32x2 xh = LN ? fma2(xp[p], rs2[j], nmr2[j]) : mul2(xp[p], rs2[j]);
              const f32x2 dyg = mul2(dp[p], gp[i][p]);
              if (LN) s1 = add2(s1, dyg);
              s2 = fma2(dyg, xh, s2);
              accg[i][p] = fma2(dp[p], xh, accg[i][p]);
              if (LN) accb[i][p] = add2(accb[i][p], dp[p]);
              xk[j][i][p] = xh;
              gk[j][i][p] = dyg;
            }
          }
        }
      }
      t1[j] = LN ? f2lo(s1) + f2hi(s1) : 0.0f;
      t2[j] = f2lo(s2) + f2hi(s2);
    }
    // the slots are no longer read
    __syncwarp();
    if (lane == 0 && ok) {
#pragma unroll
      for (int j = 0; j < RB; ++j)
        if (j < nr) mbar_arrive(smem_u32(&empty[s0 + j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
      for (int j = 0; j < RB; ++j) {
        if (LN) t1[j] += __shfl_xor_sync(0xffffffffu, t1[j], o);
        t2[j] += __shfl_xor_sync(0xffffffffu, t2[j], o);
      }
    }
    const int par = int(it & 1);
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < RB; ++j) red[par][j][warp] = make_float2(t1[j], t2[j]);
    }
    if (group_sync_or(!ok, 1, GT)) break;
    // Every warp has released the step's slots before the barrier: each slot is refilled with
    // the row spc ahead by one warp (a different one for each row, in turn), which waits on the
    // slot's empty barrier to acquire the other warps' reads.  (A failed wait has raised the
    // abort flag: the next acquire of every warp gives up.)
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      const int s = s0 + j;
      const int64_t next = j0 + j + spc;
      if (warp == int((it * RB + j) % G) && lane == 0 && j < nr && next < nloc &&
          (mbar_try_wait(smem_u32(&empty[s]), use & 1u) ||
           wait_bounded(smem_u32(&empty[s]), use & 1u, abort_flag, status, kWaitLimitNs, true))) {
        ring_issue(xsrc, dzsrc, row_bytes, next, s, ring, full);
        last_use[s] = int(use) + 1;
      }
    }
    // the warps add their sums in warp order (the same bits in every thread);
    // dx = rs * (dz * g - mean(dz * g) - xhat * mean(dz * g * xhat))
    //    = (dz * g) * rs + c1 + xhat * c2,  c1 = -rs * mean(dz * g), c2 = -rs * mean(dz * g * xhat)
#pragma unroll
    for (int j = 0; j < RB; ++j) {
      float r1 = 0.0f, r2 = 0.0f;
#pragma unroll
      for (int w = 0; w < G; ++w) {
        const float2 r = red[par][j][w];
        r1 += r.x;
        r2 += r.y;
      }
      const float rs = f2lo(rs2[j]);
      const f32x2 c1 = f2s(LN ? -rs * (r1 * inv_h) : 0.0f);
      const f32x2 c2 = f2s(-rs * (r2 * inv_h));
      // pass 2, from registers
      if (j < nr) {
        T* dxr = dx0 + j * dx_step;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
          if (mine(gt + i * GT)) {
            float d[E];
#pragma unroll
            for (int p = 0; p < P; ++p) {
              const f32x2 dd = fma2(xk[j][i][p], c2, fma2(gk[j][i][p], rs2[j], c1));
              d[2 * p] = f2lo(dd);
              d[2 * p + 1] = f2hi(dd);
            }
            store_out<(E == 8 ? OUT_BF16 : OUT_F32), E>(dxr, int64_t(i) * GT * E, d, CastState{});
          }
        }
      }
    }
    jj += RB;
    if (jj == spc) { jj = 0; ++use; }
  }
  // After a failed wait, copies issued but never consumed may still be in flight: wait for
  // them (briefly) before the CTA exits.  Without a failure every issued row was consumed.
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) {
    for (int s = 0; s < spc; ++s)
      if (last_use[s] >= 0)
        wait_bounded(smem_u32(&full[s]), uint32_t(last_use[s]) & 1u, nullptr, status,
                     kDrainLimitNs, false);
  }
  float* pg = a.partials + int64_t(blockIdx.x) * 2 * a.H;
  float* pb = pg + a.H;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = gt + i * GT;
    if (mine(v)) {
      float4* g4 = reinterpret_cast<float4*>(pg + int64_t(v) * E);
      float4* b4 = reinterpret_cast<float4*>(pb + int64_t(v) * E);
#pragma unroll
      for (int q = 0; q < P / 2; ++q) {
        g4[q] = make_float4(f2lo(accg[i][2 * q]), f2hi(accg[i][2 * q]), f2lo(accg[i][2 * q + 1]),
                            f2hi(accg[i][2 * q + 1]));
        b4[q] = make_float4(f2lo(accb[i][2 * q]), f2hi(accb[i][2 * q]), f2lo(accb[i][2 * q + 1]),
                            f2hi(accb[i][2 * q + 1]));
      }
    }
  }
}

// dgamma[j] = sum_c partials[c][0][j], dbeta[j] = sum_c partials[c][1][j].  A CTA takes 128
// columns, 4 per thread of a warp (16-byte loads); its 16 warps take the chunks c = w, w + 16,
// ... each in chunk order, and then the warps' sums are added in warp order: the same order for
// every column and every run.  (One thread per column looping over all chunks made a chain of
// about 150 dependent loads, longer than the ring kernel's own tail.)
constexpr int kRedWarps = 16;
__global__ void __launch_bounds__(kRedWarps * 32) norm_bwd_reduce_kernel(const float* partials,
                                                                         int chunks, int64_t H,
                                                                         float* dgamma,
                                                                         float* dbeta) {
  __shared__ float4 sg[kRedWarps][32], sb[kRedWarps][32];
  // launched as a programmatic dependent of the ring kernel: wait here until that grid has
  // completed and its partial sums are visible (a no-op for an ordinary launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t j = int64_t(blockIdx.x) * 128 + lane * 4;  // H is a multiple of 8
  float4 ag = make_float4(0.0f, 0.0f, 0.0f, 0.0f), ab = ag;
  if (j < H) {
#pragma unroll 4
    for (int c = w; c < chunks; c += kRedWarps) {
      const float* row = partials + int64_t(c) * 2 * H + j;
      const float4 g = *reinterpret_cast<const float4*>(row);
      const float4 b = *reinterpret_cast<const float4*>(row + H);
      ag.x += g.x; ag.y += g.y; ag.z += g.z; ag.w += g.w;
      ab.x += b.x; ab.y += b.y; ab.z += b.z; ab.w += b.w;
    }
  }
  sg[w][lane] = ag;
  sb[w][lane] = ab;
  __syncthreads();
  if (w == 0 && j < H) {
    float4 tg = sg[0][lane], tb = sb[0][lane];
#pragma unroll
    for (int v = 1; v < kRedWarps; ++v) {
      const float4 g = sg[v][lane], b = sb[v][lane];
      tg.x += g.x; tg.y += g.y; tg.z += g.z; tg.w += g.w;
      tb.x += b.x; tb.y += b.y; tb.z += b.z; tb.w += b.w;
    }
    dgamma[j] = tg.x; dgamma[j + 1] = tg.y; dgamma[j + 2] = tg.z; dgamma[j + 3] = tg.w;
    if (dbeta) { dbeta[j] = tb.x; dbeta[j + 1] = tb.y; dbeta[j + 2] = tb.z; dbeta[j + 3] = tb.w; }
  }
}

// CTAs of the backward on one SM: kBwdWarps / G.  Each takes an equal share of the SM's shared
// memory for its ring.
constexpr size_t kBwdSmPerSm = 227 * 1024;  // dynamic shared memory all CTAs of an SM may hold

int64_t bwd_grid(int64_t M, int ctas_per_sm) {
  const int64_t n = int64_t(num_sms()) * ctas_per_sm;
  return M < n ? (M > 0 ? M : 1) : n;
}

// Partial dgamma / dbeta rows: one per CTA (at most two CTAs per SM).
int bwd_chunks(int64_t M) { return int(bwd_grid(M, 2)); }

template <typename T, bool LN, int NV, bool FULL, int G>
te_status launch_bwd_t(const NormBwdArgs& a, cudaStream_t s) {
  static PerDevice<bool> attr_done;
  constexpr int RB = bwd_rows_per_sync(NV);
  constexpr int kCtas = kBwdWarps / G;
  const size_t slot_bytes = size_t(a.H) * sizeof(T) * 2;
  // a step holds RB slots; a second step's worth lets the refills run ahead
  const size_t cap = kCtas == 1 ? kRingSmemMax : kBwdSmPerSm / kCtas - 1024;
  const int spc = ring_slots(slot_bytes, kBwdMaxSlots, 2 * RB, RB, cap);
  if (spc == 0) return TE_ERR_UNSUPPORTED;
  const size_t smem = ring_header_bytes(spc) + size_t(spc) * slot_bytes;
  const te_status st = allow_ring_smem(norm_bwd_ring_kernel<T, LN, NV, FULL, G>, attr_done, kCtas > 1);
  if (st != TE_OK) return st;
  const unsigned grid = unsigned(bwd_grid(a.M, kCtas));
  norm_bwd_ring_kernel<T, LN, NV, FULL, G><<<grid, G * 32, smem, s>>>(
      a, device_status_ptr(), spc);
  if (cudaGetLastError() != cudaSuccess) return TE_ERR_CUDA;
  // the column sums: their launch overlaps the ring kernel's tail (griddepcontrol.wait in the
  // kernel orders them after the whole ring grid)
  return launch_dependent(norm_bwd_reduce_kernel, dim3(unsigned(ceil_div(a.H, 128))),
                          dim3(kRedWarps * 32), s, static_cast<const float*>(a.partials),
                          int(grid), int64_t(a.H), a.dgamma, a.dbeta);
}

template <typename T, int NV, int G>
te_status launch_bwd_nv(const NormBwdArgs& a, cudaStream_t s) {
  const bool full = a.H / Vec16<T>::N == int64_t(NV) * G * 32;
  if (a.norm_type == TE_LAYERNORM)
    return full ? launch_bwd_t<T, true, NV, true, G>(a, s) : launch_bwd_t<T, true, NV, false, G>(a, s);
  return full ? launch_bwd_t<T, false, NV, true, G>(a, s) : launch_bwd_t<T, false, NV, false, G>(a, s);
}

// Rows of up to 512 vectors (8 KB) go to two CTAs of 4 warps per SM, each thread holding up to
// 4 vectors of a row; longer rows (up to 1024 vectors, 16 KB) to one CTA of 8 warps.  Four
// vectors per thread per row keep the per-row barrier and ring bookkeeping small against the
// row's arithmetic, and two CTAs keep two rows in work per SM: LayerNorm at 16384 x 4096 went
// from 78% to 84% of the measured copy bandwidth, at 16384 x 2048 / 1024 by a third / a half.
// RMSNorm rows of 257 .. 512 vectors (less arithmetic per element) measured 1% faster with one
// CTA of 8 warps and keep it.
template <typename T>
te_status launch_bwd_dispatch(const NormBwdArgs& a, cudaStream_t s) {
  constexpr int E = Vec16<T>::N;
  const int64_t nvec = a.H / E;
  const int64_t two_cta_max = a.norm_type == TE_LAYERNORM ? 4 * 4 * 32 : 2 * 4 * 32;
  if (nvec <= two_cta_max) {
    const int64_t per_thread = ceil_div(nvec, int64_t(4 * 32));
    if (per_thread <= 1) return launch_bwd_nv<T, 1, 4>(a, s);
    if (per_thread <= 2) return launch_bwd_nv<T, 2, 4>(a, s);
    return launch_bwd_nv<T, 4, 4>(a, s);
  }
  if (nvec <= 2 * kBwdWarps * 32) return launch_bwd_nv<T, 2, kBwdWarps>(a, s);
  if (nvec <= 4 * kBwdWarps * 32) return launch_bwd_nv<T, 4, kBwdWarps>(a, s);
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
  return size_t(bwd_chunks(M)) * 2 * size_t(H) * sizeof(float);
}

te_status launch_norm_bwd(const NormBwdArgs& a, cudaStream_t s) {
  if (a.M == 0) return TE_OK;
  ProfileScope prof(TE_KERNEL_NORM_BWD, s);
  if (a.dtype == TE_BF16) return launch_bwd_dispatch<__nv_bfloat16>(a, s);
  if (a.dtype == TE_F32) return launch_bwd_dispatch<float>(a, s);
  return TE_ERR_UNSUPPORTED;
}

}  // namespace te
