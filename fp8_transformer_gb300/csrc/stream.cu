// Streaming kernels for the activation (act_lu) and the backward's activation gradient + bias
// reduction + quantize (dact_dbias), fed by TMA.
//
// TransformerEngine JAX "Activation" page (Description: the forward rule's activation
// primitive with optional FP8 round trip) and "LayerNorm MLP" page (Description, backward: the
// fused quantize / dact / dbias primitive).
//
// Layout of the work: the [M, n] problem is cut into items of one 512-byte column strip (32
// lanes x 16 bytes) by 128 rows.  A CTA (persistent, two per SM) has one producer warp and 8
// consumer warps.  The producer streams each input's 16-row x 512-byte tiles of the current
// item into a 4-stage shared-memory ring (up to 24 KB a stage, so ~100 KB in flight per CTA
// without holding anything in registers); consumer warp w takes rows w and w + 8 of every
// stage, computes on f32x2 pairs and stores its results with coalesced 16-byte stores.  For
// the bias gradient each consumer thread sums its 8 columns over the item's rows in registers;
// at the end of the item the 8 warps combine through shared memory in warp order and write one
// partial row, and an ordered second kernel adds the partial rows, so dbias is deterministic.
// Every wait (the ring and the end-of-item combine) is a bounded mbarrier wait.
#include <cstdlib>
#include <cstring>

#include "cast.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace te {
namespace {

constexpr int kSWarps = 8;                      // consumer warps
constexpr int kSThreads = 32 * (kSWarps + 1);   // + the producer warp
constexpr int kSRows = 16;                      // rows per stage
constexpr int kSStages = 4;
constexpr int kItemRows = 128;                  // rows per item = rows per dbias partial
constexpr int kSRowBytes = 512;                 // one row of a strip
constexpr int kSTile = kSRows * kSRowBytes;     // 8 KB
constexpr int kSMaxTiles = 3;                   // dy, x (gate), linear half

struct StreamParams {
  CUtensorMap tm_dy;  // [M, n_out]  (dact only)
  CUtensorMap tm_x;   // [M, N_in]
  int dact;           // 0: act_lu, 1: dact_dbias
  int act;
  int gated, ident;
  int64_t M, N_in, n_out;
  void* out;          // act: [M, n_out]; dact: dx [M, N_in] or null
  float* dbias;       // dact: non-null -> write partial rows
  float* partials;    // [ceil(M / 128), N_in]
  CastSpec cast;
  int num_strips, num_items;
  int ntiles;         // tiles per stage
  int* status;
};

constexpr size_t kSmemRing = size_t(kSStages) * kSMaxTiles * kSTile;           // 96 KB
constexpr size_t kSmemRed = size_t(kSWarps) * 2 * 32 * 8 * sizeof(float);      // 16 KB
constexpr size_t kSmemBytes = kSmemRing + kSmemRed + 128;

template <typename T>
__global__ void __launch_bounds__(kSThreads, 2) stream_kernel(const __grid_constant__ StreamParams p) {
  using V = Vec16<T>;
  using PR = Pairs<T>;
  constexpr int E = V::N;
  constexpr int P = PR::P;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  float* red = reinterpret_cast<float*>(smem + kSmemRing);  // [kSWarps][2][32 * E]
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemRing + kSmemRed);
  uint64_t* full = bars;                 // [kSStages]
  uint64_t* empty = bars + kSStages;     // [kSStages]
  uint64_t* red_full = bars + 2 * kSStages;
  uint64_t* red_empty = red_full + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kSStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kSWarps);
    }
    mbar_init(smem_u32(red_full), kSWarps * 32);
    mbar_init(smem_u32(red_empty), kSWarps * 32);
    mbar_init_fence();
  }
  __syncthreads();
  const int64_t n_out = p.n_out;
  const uint32_t stage_bytes = uint32_t(p.ntiles) * kSTile;

  if (warp == kSWarps) {
    // ------------------------------------------------------------ producer -------------
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < p.num_items && ok; w += gridDim.x) {
        const int strip = w % p.num_strips;
        const int64_t r0 = int64_t(w / p.num_strips) * kItemRows;
        const int64_t r1 = r0 + kItemRows < p.M ? r0 + kItemRows : p.M;
        const int col = strip * 32 * E;
        for (int64_t r = r0; r < r1; r += kSRows) {
          if (!mbar_try_wait(smem_u32(&empty[stage]), phase ^ 1) &&
              !wait_bounded(smem_u32(&empty[stage]), phase ^ 1, nullptr, p.status, kWaitLimitNs, false)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_expect_tx(fb, stage_bytes);
          const uint32_t dst = smem_u32(ring + size_t(stage) * kSMaxTiles * kSTile);
          int t = 0;
          if (p.dact) tma_load_2d(dst + (t++) * kSTile, &p.tm_dy, fb, col, int(r));
          if (!p.ident) tma_load_2d(dst + (t++) * kSTile, &p.tm_x, fb, col, int(r));
          if (p.gated) tma_load_2d(dst + (t++) * kSTile, &p.tm_x, fb, int(n_out) + col, int(r));
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == kSStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      for (int s = 0; s < kSStages; ++s)
        if (issued & (1u << s))
          wait_bounded(smem_u32(&full[s]), (last_parity >> s) & 1, nullptr, p.status, kDrainLimitNs, false);
    }
  } else {
    // ------------------------------------------------------------ consumers ------------
    const CastState cs = cast_begin(p.cast);
    int stage = 0;
    uint32_t phase = 0, item_phase = 0;
    float amax = 0.0f;
    bool ok = true;
    for (int w = blockIdx.x; w < p.num_items && ok; w += gridDim.x, item_phase ^= 1) {
      const int strip = w % p.num_strips;
      const int64_t rg = w / p.num_strips;
      const int64_t r0 = rg * kItemRows;
      const int64_t r1 = r0 + kItemRows < p.M ? r0 + kItemRows : p.M;
      const int64_t col = int64_t(strip) * 32 * E + int64_t(lane) * E;
      const bool valid = col < n_out;
      f32x2 acc1[P], acc2[P];
#pragma unroll
      for (int q = 0; q < P; ++q) { acc1[q] = f2s(0.0f); acc2[q] = f2s(0.0f); }
      for (int64_t r = r0; r < r1; r += kSRows) {
        const uint32_t fb = smem_u32(&full[stage]);
        int got = 1;
        if (lane == 0) got = (mbar_try_wait(fb, phase) ||
                              wait_bounded(fb, phase, nullptr, p.status, kWaitLimitNs, false)) ? 1 : 0;
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        while (!mbar_try_wait(fb, phase)) {
        }
        __syncwarp();
        const uint8_t* tiles = ring + size_t(stage) * kSMaxTiles * kSTile;
        const int t_x = p.dact ? 1 : 0;
#pragma unroll
        for (int jj = 0; jj < kSRows / kSWarps; ++jj) {
          const int j = warp + jj * kSWarps;
          const int64_t row = r + j;
          if (row >= r1 || !valid) continue;
          const size_t off = size_t(j) * kSRowBytes + size_t(lane) * 16;
          f32x2 hp[P], lp[P], dyp[P];
          if (!p.ident) PR::get(*reinterpret_cast<const uint4*>(tiles + t_x * kSTile + off), hp);
          if (p.gated) PR::get(*reinterpret_cast<const uint4*>(tiles + (t_x + 1) * kSTile + off), lp);
          float y1[E], y2[E];
          if (!p.dact) {
#pragma unroll
            for (int q = 0; q < P; ++q) {
              const f32x2 yy = p.gated ? mul2(silu2(hp[q]), lp[q]) : act2(p.act, hp[q]);
              amax = absmax2(amax, yy);
              y1[2 * q] = f2lo(yy);
              y1[2 * q + 1] = f2hi(yy);
            }
            if (cs.store) cast_store<E>(p.out, row * n_out + col, y1, cs);
          } else {
            PR::get(*reinterpret_cast<const uint4*>(tiles + off), dyp);
            if (p.gated) {
#pragma unroll
              for (int q = 0; q < P; ++q) {
                f32x2 sg, eg;
                sigmoid2(hp[q], sg, eg);
                const f32x2 dsil = mul2(sg, fma2(hp[q], mul2(eg, sg), f2s(1.0f)));
                const f32x2 g2 = mul2(mul2(dyp[q], lp[q]), dsil);
                const f32x2 l2 = mul2(dyp[q], mul2(hp[q], sg));
                acc1[q] = add2(acc1[q], g2);
                acc2[q] = add2(acc2[q], l2);
                amax = absmax2(absmax2(amax, g2), l2);
                y1[2 * q] = f2lo(g2);
                y1[2 * q + 1] = f2hi(g2);
                y2[2 * q] = f2lo(l2);
                y2[2 * q + 1] = f2hi(l2);
              }
              if (cs.store) {
                cast_store<E>(p.out, row * p.N_in + col, y1, cs);
                cast_store<E>(p.out, row * p.N_in + n_out + col, y2, cs);
              }
            } else {
#pragma unroll
              for (int q = 0; q < P; ++q) {
                const f32x2 dd = p.ident ? dyp[q] : mul2(dyp[q], dact2(p.act, hp[q]));
                acc1[q] = add2(acc1[q], dd);
                amax = absmax2(amax, dd);
                y1[2 * q] = f2lo(dd);
                y1[2 * q + 1] = f2hi(dd);
              }
              if (cs.store && p.out) cast_store<E>(p.out, row * p.N_in + col, y1, cs);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[stage]));
        if (++stage == kSStages) {
          stage = 0;
          phase ^= 1;
        }
      }
      if (!ok || !p.dbias) continue;
      // Combine the 8 warps' column sums for this item in warp order.  red_empty guards the
      // reuse of `red` by the next item; both waits are bounded.
      const uint32_t re = smem_u32(red_empty), rf = smem_u32(red_full);
      if (!(mbar_try_wait(re, item_phase ^ 1) ||
            wait_bounded(re, item_phase ^ 1, nullptr, p.status, kWaitLimitNs, false))) {
        ok = false;
        break;
      }
      float* mine = red + size_t(warp) * 2 * 32 * E;
#pragma unroll
      for (int q = 0; q < P; ++q) {
        mine[lane * E + 2 * q] = f2lo(acc1[q]);
        mine[lane * E + 2 * q + 1] = f2hi(acc1[q]);
        mine[32 * E + lane * E + 2 * q] = f2lo(acc2[q]);
        mine[32 * E + lane * E + 2 * q + 1] = f2hi(acc2[q]);
      }
      mbar_arrive(rf);
      if (!(mbar_try_wait(rf, item_phase) ||
            wait_bounded(rf, item_phase, nullptr, p.status, kWaitLimitNs, false))) {
        ok = false;
        break;
      }
      const int halves = p.gated ? 2 : 1;
      for (int t = threadIdx.x; t < halves * 32 * E; t += kSWarps * 32) {
        const int hsel = t / (32 * E), jcol = t % (32 * E);
        float sum = 0.0f;
#pragma unroll
        for (int w2 = 0; w2 < kSWarps; ++w2) sum += red[size_t(w2) * 2 * 32 * E + hsel * 32 * E + jcol];
        const int64_t c = int64_t(strip) * 32 * E + jcol;
        if (c < n_out) p.partials[rg * p.N_in + hsel * n_out + c] = sum;
      }
      mbar_arrive(re);
    }
    amax = warp_max(amax);
    if (lane == 0 && p.cast.amax_out) atomic_max_nonneg(p.cast.amax_out, amax);
  }
  __syncthreads();
}

size_t stream_smem() { return kSmemBytes; }

template <typename T>
te_status launch_stream_t(StreamParams& p, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (!attr_set[dev & 63]) {
    if (cudaFuncSetAttribute(stream_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kSmemBytes)) != cudaSuccess)
      return TE_ERR_CUDA;
    attr_set[dev & 63] = true;
  }
  const int64_t slots = int64_t(num_sms()) * 2;
  const unsigned grid = unsigned(p.num_items < slots ? p.num_items : slots);
  stream_kernel<T><<<grid, kSThreads, kSmemBytes, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

te_status launch_stream(StreamParams& p, int dtype, const void* dy, const void* x, cudaStream_t s) {
  const int E = dtype == TE_BF16 ? 8 : 4;
  const uint32_t box_cols = uint32_t(32 * E);
  if (p.M == 0) return TE_OK;
  if (p.dact && !make_tmap_2d(&p.tm_dy, dy, dtype, uint64_t(p.n_out), uint64_t(p.M), box_cols, kSRows, false))
    return TE_ERR_CUDA;
  if (!p.ident && !make_tmap_2d(&p.tm_x, x, dtype, uint64_t(p.N_in), uint64_t(p.M), box_cols, kSRows, false))
    return TE_ERR_CUDA;
  p.num_strips = int(ceil_div(p.n_out, 32 * E));
  const int64_t items = int64_t(p.num_strips) * ceil_div(p.M, kItemRows);
  if (items > 0x7fffffff) return TE_ERR_UNSUPPORTED;
  p.num_items = int(items);
  p.ntiles = (p.dact ? 1 : 0) + (p.ident ? 0 : 1) + (p.gated ? 1 : 0);
  p.status = device_status_ptr();
  if (dtype == TE_BF16) return launch_stream_t<__nv_bfloat16>(p, s);
  if (dtype == TE_F32) return launch_stream_t<float>(p, s);
  return TE_ERR_UNSUPPORTED;
}

__global__ void colsum_partials_kernel(const float* partials, int chunks, int64_t n, float* out) {
  const int64_t j = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= n) return;
  float s = 0.0f;
  for (int c = 0; c < chunks; ++c) s += partials[int64_t(c) * n + j];
  out[j] = s;
}

}  // namespace

bool use_tma_streams() {
  static int v = -1;
  if (v < 0) {
    const char* e = getenv("TE_STREAM_TMA");
    v = (e && e[0] == '1') ? 1 : 0;
  }
  return v == 1;
}

te_status launch_act_lu(const ActArgs& a, cudaStream_t s) {
  ProfileScope prof(TE_KERNEL_ACT_LU, s);
  if (a.x_dtype != TE_BF16 && a.x_dtype != TE_F32) return TE_ERR_UNSUPPORTED;
  if (!use_tma_streams()) return launch_act_lu_reg(a, s);
  StreamParams p;
  memset(&p, 0, sizeof(p));
  p.dact = 0;
  p.act = a.act;
  p.gated = a.act == TE_SWIGLU;
  p.ident = 0;
  p.M = a.M;
  p.N_in = a.N_in;
  p.n_out = p.gated ? a.N_in / 2 : a.N_in;
  p.out = a.out;
  p.cast = a.cast;
  return launch_stream(p, a.x_dtype, nullptr, a.x, s);
}

size_t dact_dbias_workspace(int64_t M, int64_t N_in) {
  return size_t(ceil_div(M > 0 ? M : 1, kItemRows)) * size_t(N_in) * sizeof(float);
}

te_status launch_dact_dbias(const DactArgs& a, cudaStream_t s) {
  if (a.M == 0) return TE_OK;
  ProfileScope prof(TE_KERNEL_DACT_DBIAS, s);
  if (a.dtype != TE_BF16 && a.dtype != TE_F32) return TE_ERR_UNSUPPORTED;
  StreamParams p;
  memset(&p, 0, sizeof(p));
  p.dact = 1;
  p.act = a.act;
  p.gated = a.act == TE_SWIGLU;
  p.ident = a.act == TE_IDENTITY;
  p.M = a.M;
  p.N_in = a.N_in;
  p.n_out = p.gated ? a.N_in / 2 : a.N_in;
  p.out = a.dx;
  p.dbias = a.dbias;
  p.partials = a.partials;
  p.cast = a.cast;
  te_status st = use_tma_streams() ? launch_stream(p, a.dtype, a.dy, a.x, s) : launch_dact_reg(a, s);
  if (st != TE_OK || !a.dbias) return st;
  const int chunks = int(ceil_div(a.M, kItemRows));
  colsum_partials_kernel<<<unsigned(ceil_div(a.N_in, 256)), 256, 0, s>>>(a.partials, chunks,
                                                                         a.N_in, a.dbias);
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

}  // namespace te
