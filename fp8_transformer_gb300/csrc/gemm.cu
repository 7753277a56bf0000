// Tensor-core GEMM with fused epilogues for sm_103a: TMA -> shared-memory ring -> tcgen05.mma
// into a double-buffered TMEM accumulator -> tcgen05.ld epilogue.
//
// It implements the two bias-carrying GEMMs of the TransformerEngine JAX "LayerNorm MLP" page
// (Description, forward steps (2) and (4)) and the one GEMM of the "LayerNorm Dense" page, with
// the activation and FP8 cast of step (3) fused into the first GEMM's epilogue.
//
// Structure (persistent over output tiles; by default clusters of two CTAs on an SM pair
// compute 256 x 256 tiles with tcgen05.mma.cta_group::2, one CTA per SM):
//   warp 0     TMA producer: one elected thread fills a STAGES-deep ring of A/B tiles, each
//              row of a tile 128 bytes of K in the 128-byte swizzled layout (each CTA of a
//              pair loads its own 128 rows of A and its half of the tile's B columns).
//   warp 1     owns the TMEM allocation (512 columns = two 256-column fp32 accumulators) and,
//              in the pair's even CTA, issues tcgen05.mma from one thread; tcgen05.commit
//              releases ring slots (multicast to both CTAs) and hands a finished accumulator to
//              the epilogue.
//   warps 2-9  epilogue, two warps per TMEM lane quadrant: tcgen05.ld 32 columns at a time,
//              scale by the FP8 dequantization factor, add the bias, round the pre-activation,
//              apply the activation (a gated pair's gate and linear halves sit in the two
//              column halves of one accumulator tile), track amax, and store fp32 / bf16 /
//              E4M3.
// The epilogue of tile i overlaps the MMAs of tile i + 1.  Tiles go in raster groups of m-tiles
// that keep their A rows in L2; a B of at most 64 MB is instead kept in L2 for the whole GEMM
// (n fastest, with L2 eviction hints on the loads) while A streams through once.
//
// When the tiles do not fill the last wave of SM pairs, and the caller gives scratch memory, the
// tiles of that wave are split along K into chunks computed by different pairs: every chunk
// stores its raw fp32 accumulator, and the pair whose chunk is counted in last sums them in
// chunk order (so the result is the same whichever pair finishes last) and runs the epilogue.
//
// Every mbarrier wait is bounded in time.  On expiry the waiting thread records
// TE_ERR_TIMEOUT in the device status word and raises a CTA-wide abort flag; every role
// then leaves its loop, the producer waits (again bounded) for its own TMA copies still in
// flight, the MMA thread waits for its own MMAs, and TMEM is freed before the CTA exits.
#include <cuda.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "sync.cuh"

namespace te {

__device__ int g_device_status;

namespace {

constexpr int BM = 128;                 // accumulator rows per CTA (TMEM lanes)
constexpr int BN = 256;                 // accumulator columns per tile
constexpr int kRowBytes = 128;          // bytes of K per tile row per stage

// CG = CTAs per MMA (tcgen05 cta_group).  CG == 2: a cluster of two CTAs on two SMs computes a
// 256 x 256 tile; each CTA holds 128 rows of A and 128 columns of B, so each SM streams and
// reads half of B per MMA.
template <int CG>
struct Cfg {
  static constexpr int kBRows = BN / CG;                // B columns held per CTA
  static constexpr int kStages = CG == 1 ? 4 : 6;
  static constexpr int kAStage = BM * kRowBytes;        // 16 KB
  static constexpr int kBStage = kBRows * kRowBytes;    // 32 KB or 16 KB
  static constexpr size_t kSmem = size_t(kStages) * (kAStage + kBStage) + 1024 + 256;
};
constexpr int kEpiWarps = 8;               // two warps per TMEM lane quadrant
constexpr int kThreads = 32 * (2 + kEpiWarps);  // producer, MMA, epilogue warps
constexpr uint32_t kTmemCols = 512;
constexpr int64_t kRasterL2Bytes = 48ll << 20;  // A rows a raster group may keep in L2
constexpr int64_t kBResidentBytes = 64ll << 20; // largest B kept in L2 by the n-major raster

// Element kinds: 0 = bf16 (kind::f16), 1 = E4M3 (kind::f8f6f4), 2 = fp32 as tf32 (kind::tf32).
template <int KIND>
struct Kind;
template <> struct Kind<0> { static constexpr int esize = 2; static constexpr uint32_t fmt = 1; };
template <> struct Kind<1> { static constexpr int esize = 1; static constexpr uint32_t fmt = 0; };
template <> struct Kind<2> { static constexpr int esize = 4; static constexpr uint32_t fmt = 2; };

struct GemmDev {
  int64_t M, N, K;
  int num_m, num_n, num_kb;
  int group_m;      // m-tiles per raster group (m-major raster)
  int n_major;      // B-resident raster: n fastest over every n-tile, A loads evict-first and
                    // B loads evict-last in L2
  int gated;
  int64_t F;        // gated: column offset of the linear half in B
  int epilogue, act;
  const float* a_scale_inv;
  const float* b_scale_inv;
  const void* bias;
  int bias_dtype;
  int h_dtype;
  void* saved_h;
  void* D;
  int d_dtype;
  const float* out_scale;
  float* out_scale_inv;
  float* amax_out;
  int* status;
  // The tiles after the first `full_tiles` (the last, partial wave) are split along K into
  // `split` chunks of `kb_chunk` k-blocks; chunks 0 .. split-2 leave their raw accumulators in
  // `partials` and count themselves in `flags` (zeroed before the launch); the last chunk's
  // CTA adds them to its own and runs the epilogue.
  int full_tiles;
  int split;
  int kb_chunk;
  float* partials;  // [remaining tiles][split - 1][CG][BM][BN]
  int* flags;       // [remaining tiles][CG]
};

struct GemmParams {  // aligned like its tensor maps
  CUtensorMap tmA;
  CUtensorMap tmB;
  GemmDev g;
};

// ------------------------------------------------------------------ PTX wrappers ----------

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: 128-byte swizzle, descriptor version 1 (bits 46-48).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor: fp32 accumulator, A/B format, operand majors, N >> 3, M >> 4.
template <int KIND, int CG>
__host__ __device__ constexpr uint32_t instr_desc(int a_mn_major, int b_mn_major) {
  return (1u << 4) | (Kind<KIND>::fmt << 7) | (Kind<KIND>::fmt << 10) |
         (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(BN >> 3) << 17) | (uint32_t((BM * CG) >> 4) << 24);
}

#define TE_UMMA_ASM(CGS, KINDS)                                                          \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                          \
               "tcgen05.mma.cta_group::" CGS ".kind::" KINDS " [%0], %1, %2, %3, p;\n\t}" ::"r"( \
                   d_tmem),                                                                \
               "l"(a), "l"(b), "r"(idesc), "r"(accumulate))

template <int KIND, int CG>
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  if constexpr (CG == 1) {
    if constexpr (KIND == 0) TE_UMMA_ASM("1", "f16");
    else if constexpr (KIND == 1) TE_UMMA_ASM("1", "f8f6f4");
    else TE_UMMA_ASM("1", "tf32");
  } else {
    if constexpr (KIND == 0) TE_UMMA_ASM("2", "f16");
    else if constexpr (KIND == 1) TE_UMMA_ASM("2", "f8f6f4");
    else TE_UMMA_ASM("2", "tf32");
  }
}
#undef TE_UMMA_ASM

// Arrives on `bar` (this CTA) once every tcgen05.mma issued so far by this thread completed.
template <int CG>
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
  else
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Same, arriving on the barrier at this offset in every CTA of `mask` (cluster of two).
__device__ __forceinline__ void umma_commit_mc(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}

template <int CG>
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t cols) {
  if constexpr (CG == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int CG>
__device__ __forceinline__ void tmem_dealloc(uint32_t base, uint32_t cols) {
  if constexpr (CG == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols)
                 : "memory");
}

// TMA load whose completion is signaled on an mbarrier that may sit in the peer CTA of the
// pair (`bar` is a shared::cluster address).
// The same loads with an L2 eviction priority (a policy from createpolicy).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* tm, uint32_t bar,
                                                 int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint(uint32_t dst, const CUtensorMap* tm,
                                                      uint32_t bar, int c0, int c1, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* tm, uint32_t bar,
                                                 int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// shared::cluster address of the same shared-memory offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread t of the warp receives its TMEM lane's row.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Stores 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// TMEM column of the k-th (of 4) 32-column group an epilogue warp of column half `half` reads:
// one half of the tile, or for a gated tile the matching quarter of each of its two halves.
__device__ __forceinline__ int epilogue_column(int k, int half, int gated) {
  if (!gated) return (half * 4 + k) * 32;
  return (k >> 1) * (BN / 2) + (half * 2 + (k & 1)) * 32;
}

// ------------------------------------------------------------------ tile order ------------

struct Tile {
  int m, n;
};

// Raster groups of group_m m-tiles, m fastest: the tiles in flight share B columns, and a
// group's A rows stay in L2 while the group sweeps every n column.  n_major: n fastest over all
// n-tiles, one m row of tiles after another, for a B small enough to stay in L2 for the whole
// GEMM while A streams through once.
__device__ __forceinline__ Tile tile_of(int t, int num_m, int num_n, int group_m, int n_major) {
  if (n_major) return Tile{t / num_n, t % num_n};
  const int group_size = group_m * num_n;
  const int group = t / group_size;
  const int first_m = group * group_m;
  const int gm = min(num_m - first_m, group_m);
  const int in_group = t - group * group_size;
  return Tile{first_m + in_group % gm, in_group / gm};
}

// A cluster's unit of work: tile `tile`, k-blocks [kb0, kb1), and which K chunk of a split
// tile it is (-1: the whole tile).  Items [0, full_tiles) are whole tiles in raster order; the
// rest are the remaining tiles' chunks, chunk-minor, so a tile's last chunk comes after its
// other chunks in every cluster's sequence.
struct Item {
  int tile, kb0, kb1, chunk;
};

__device__ __forceinline__ Item item_of(int it, const GemmDev& g) {
  if (it < g.full_tiles) return Item{it, 0, g.num_kb, -1};
  const int u = it - g.full_tiles;
  const int c = u % g.split;
  const int kb0 = c * g.kb_chunk;
  const int kb1 = kb0 + g.kb_chunk < g.num_kb ? kb0 + g.kb_chunk : g.num_kb;
  return Item{g.full_tiles + u / g.split, kb0, kb1, g.split > 1 ? c : -1};
}

// Counts a split tile's chunks in at GPU scope: releases this chunk's partial, acquires the
// earlier ones', returns how many chunks had arrived before.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// A K chunk's raw accumulator (one CTA's 128 x 256 fp32) in 4-column groups with the 128 rows
// contiguous, so the 32 rows of a warp's access are one 512-byte run.
__device__ __forceinline__ size_t partial_index(int col, int row) {
  return (size_t(col >> 2) * BM + row) * 4;
}

__device__ __forceinline__ void store_partial(float* base, int col, int row, const uint32_t (&r)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    __stcg(reinterpret_cast<float4*>(base + partial_index(col + 4 * j, row)),
           make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                       __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3])));
}

// r (this chunk's accumulator, columns [col, col + 32) of one row) becomes the sum of all the
// tile's chunks, added in chunk order so that the result does not depend on which chunk ran last.
template <int CG>
__device__ __forceinline__ void add_chunks(uint32_t (&r)[32], const float* slot0, int own, int split,
                                           int col, int row) {
  constexpr size_t kChunkStride = size_t(CG) * BM * BN;  // from one chunk's partials to the next's
  float t[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float4 p;
    if (own == 0) {
      p = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                      __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
    } else {
      p = __ldcg(reinterpret_cast<const float4*>(slot0 + partial_index(col + 4 * j, row)));
    }
    t[4 * j] = p.x;
    t[4 * j + 1] = p.y;
    t[4 * j + 2] = p.z;
    t[4 * j + 3] = p.w;
  }
#pragma unroll 1
  for (int c = 1; c < split; ++c) {
    if (c == own) {
#pragma unroll
      for (int i = 0; i < 32; ++i) t[i] += __uint_as_float(r[i]);
    } else {
      const float* b = slot0 + size_t(c) * kChunkStride;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 p = __ldcg(reinterpret_cast<const float4*>(b + partial_index(col + 4 * j, row)));
        t[4 * j] += p.x;
        t[4 * j + 1] += p.y;
        t[4 * j + 2] += p.z;
        t[4 * j + 3] += p.w;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(t[i]);
}

// ------------------------------------------------------------------ epilogue stores -------

__device__ __forceinline__ void store_seg(void* base, int64_t off, const float (&v)[32],
                                          int count, int dtype, float scale) {
  if (dtype == TE_F32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i * 4 < count) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  } else if (dtype == TE_BF16) {
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(base) + off);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (i * 8 < count)
        p[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16x2(v[8 * i + 4], v[8 * i + 5]),
                          pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
  } else {
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint8_t*>(base) + off);
    const f32x2 s2 = f2s(scale);
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (i * 16 < count) {
        uint32_t w4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {  // fp32(v * scale) on pairs, then the E4M3 codes
          const float* w = v + 16 * i + 4 * q;
          const f32x2 a = mul2(f2(w[0], w[1]), s2), b = mul2(f2(w[2], w[3]), s2);
          w4[q] = pack_e4m3x4(f2lo(a), f2hi(a), f2lo(b), f2hi(b));
        }
        p[i] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
      }
  }
}

// The bias values of columns j and j + 1 (j even) as an fp32 pair.
__device__ __forceinline__ f32x2 load_bias_pair(const void* bias, int dtype, int64_t j) {
  if (dtype == TE_BF16)
    return bf16x2_f2(__ldg(reinterpret_cast<const uint32_t*>(static_cast<const uint16_t*>(bias) + j)));
  const float2 w = __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(bias) + j));
  return f2(w.x, w.y);
}

// The bias of columns col0 .. col0 + 31 as fp32 pairs (zero past `count`, or without a bias).
__device__ __forceinline__ void load_bias_chunk(const void* bias, int dtype, int64_t col0,
                                                int count, f32x2 (&b)[16]) {
#pragma unroll
  for (int p = 0; p < 16; ++p)
    b[p] = (bias && 2 * p < count) ? load_bias_pair(bias, dtype, col0 + 2 * p) : f2s(0.0f);
}

// The activation applied to a chunk of 32 values, one inner loop per activation (a switch
// per chunk, none per element, so that the compiler interleaves the 16 independent pairs).
template <int ACT>
__device__ __forceinline__ void act_chunk_t(float (&v)[32]) {
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const f32x2 y = act2c<ACT>(f2(v[2 * p], v[2 * p + 1]));
    v[2 * p] = f2lo(y);
    v[2 * p + 1] = f2hi(y);
  }
}
__device__ __forceinline__ void act_chunk(int act, float (&v)[32]) {
  switch (act) {
    case TE_RELU: act_chunk_t<TE_RELU>(v); break;
    case TE_GELU: act_chunk_t<TE_GELU>(v); break;
    case TE_SILU: act_chunk_t<TE_SILU>(v); break;
    default: break;
  }
}

// A gated pair's output base(gate) * linear into vg, the base function a compile-time choice.
template <int ACT>
__device__ __forceinline__ void gated_chunk_t(float (&vg)[32], const float (&vl)[32]) {
#pragma unroll
  for (int p = 0; p < 16; ++p) {
    const f32x2 y = mul2(act2c<ACT>(f2(vg[2 * p], vg[2 * p + 1])), f2(vl[2 * p], vl[2 * p + 1]));
    vg[2 * p] = f2lo(y);
    vg[2 * p + 1] = f2hi(y);
  }
}
__device__ __forceinline__ void gated_chunk(int base_act, float (&vg)[32], const float (&vl)[32]) {
  switch (base_act) {
    case TE_RELU: gated_chunk_t<TE_RELU>(vg, vl); break;
    case TE_GELU: gated_chunk_t<TE_GELU>(vg, vl); break;
    default: gated_chunk_t<TE_SILU>(vg, vl); break;
  }
}

// Running max of |v| over the first `count` values of a chunk; a full chunk by a tree of
// depth 5 rather than a chain of 32 (the max ignores NaN and is the same in any order).
__device__ __forceinline__ float chunk_amax(float m, const float (&v)[32], int count) {
  if (count == 32) {
    float t[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) t[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
#pragma unroll
    for (int w = 8; w >= 1; w >>= 1)
#pragma unroll
      for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
    return fmaxf(m, t[0]);
  }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < count) m = fmaxf(m, fabsf(v[i]));
  return m;
}

// Rounds both halves of a pair to bf16 (round to nearest even) and back to fp32.
__device__ __forceinline__ f32x2 round_bf16_2(f32x2 v) {
  return bf16x2_f2(pack_bf16x2(f2lo(v), f2hi(v)));
}

// ------------------------------------------------------------------ the kernel ------------

template <int KIND, bool A_KMAJOR, bool B_KMAJOR, int CG>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
  using C = Cfg<CG>;
  constexpr int STAGES = C::kStages;
  constexpr int A_STAGE = C::kAStage;
  constexpr int B_STAGE = C::kBStage;
  constexpr int BROWS = C::kBRows;
  constexpr int EPR = kRowBytes / Kind<KIND>::esize;  // K elements per 128-byte row
  constexpr int MMA_K_BYTES = 32;                     // K bytes consumed by one tcgen05.mma
  constexpr int MMA_K = MMA_K_BYTES / Kind<KIND>::esize;
  constexpr uint32_t IDESC = instr_desc<KIND, CG>(A_KMAJOR ? 0 : 1, B_KMAJOR ? 0 : 1);
  const GemmDev& g = p.g;
  // the kernel after this one may launch its setup now (it waits for this grid's completion)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* smA = smem;
  uint8_t* smB = smem + STAGES * A_STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smB + STAGES * B_STAGE);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* epi_bar = drain + 1;  // barrier of the epilogue warps (split tiles)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(epi_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* split_arrival = abort_flag + 1;  // [2]: a split chunk's arrival number

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int num_tiles = g.num_m * g.num_n;
  const int num_items = g.full_tiles + (num_tiles - g.full_tiles) * g.split;
  const uint32_t rank = CG == 1 ? 0u : cluster_rank();
  const bool leader = rank == 0;
  const int cluster_id = int(blockIdx.x) / CG;
  const int num_clusters = int(gridDim.x) / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 32 * kEpiWarps * CG);
    }
    mbar_init(smem_u32(drain), 1);
    mbar_init(smem_u32(epi_bar), 32 * kEpiWarps);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmB)) : "memory");
  }
  if (warp == 1) tmem_alloc<CG>(smem_u32(tmem_slot), kTmemCols);
  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched as a programmatic dependent of the kernel before it: the setup above overlapped
  // that kernel's tail; nothing it writes (the A operand, the scales) is read before this wait.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    // ----------------------------------------------------------- TMA producer -----------
    if (lane == 0) {
      const uint64_t pol_a = l2_policy_evict_first(), pol_b = l2_policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_parity = 0;
      bool ok = true;
      for (int it = cluster_id; it < num_items && ok; it += num_clusters) {
        const Item w = item_of(it, g);
        const Tile tl = tile_of(w.tile, g.num_m, g.num_n, g.group_m, g.n_major);
        const int m0 = (tl.m * CG + int(rank)) * BM;
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_try_wait(smem_u32(&empty[stage]), phase ^ 1) &&
              !wait_bounded(smem_u32(&empty[stage]), phase ^ 1, abort_flag, &g_device_status, kWaitLimitNs, true)) {
            ok = false;
            break;
          }
          // The pair's loads all complete on the leader's full barrier.
          const uint32_t fb = CG == 1 ? smem_u32(&full[stage]) : map_to_rank(smem_u32(&full[stage]), 0);
          if (leader) mbar_expect_tx(smem_u32(&full[stage]), CG * (A_STAGE + B_STAGE));
          const uint32_t a_dst = smem_u32(smA + stage * A_STAGE);
          const uint32_t b_dst = smem_u32(smB + stage * B_STAGE);
          const int k0 = kb * EPR;
          auto load = [&](uint32_t dst, const CUtensorMap* tm, int c0, int c1) {
            if (g.n_major) {
              const uint64_t pol = tm == &p.tmA ? pol_a : pol_b;
              if constexpr (CG == 1) tma_load_2d_hint(dst, tm, fb, c0, c1, pol);
              else tma_load_2d_pair_hint(dst, tm, fb, c0, c1, pol);
            } else {
              if constexpr (CG == 1) tma_load_2d(dst, tm, fb, c0, c1);
              else tma_load_2d_pair(dst, tm, fb, c0, c1);
            }
          };
          if constexpr (A_KMAJOR) {
            load(a_dst, &p.tmA, k0, m0);
          } else {
#pragma unroll
            for (int i = 0; i < BM / EPR; ++i) load(a_dst + i * EPR * kRowBytes, &p.tmA, m0 + i * EPR, k0);
          }
          // B columns held by this CTA: [n, n + BROWS) of the tile, or for a gated tile the gate
          // half (rank 0 / first half) and the linear half (rank 1 / second half).
          const int parts = (CG == 1 && g.gated) ? 2 : 1;
#pragma unroll
          for (int h = 0; h < parts; ++h) {
            int c0;
            if (!g.gated) c0 = tl.n * BN + int(rank) * BROWS;
            else c0 = int((CG == 1 ? h : int(rank)) * g.F) + tl.n * (BN / 2);
            const int cols = g.gated ? BN / 2 : BROWS;
            const uint32_t dst = b_dst + h * (BN / 2) * kRowBytes;
            if constexpr (B_KMAJOR) {
              load(dst, &p.tmB, k0, c0);
            } else {
              for (int i = 0; i < cols / EPR; ++i) load(dst + i * EPR * kRowBytes, &p.tmB, c0 + i * EPR, k0);
            }
          }
          issued |= 1u << stage;
          last_parity = (last_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (leader) {
        // Copies still in flight (the pair's) complete before the CTAs may exit.
        for (int s = 0; s < STAGES; ++s)
          if (issued & (1u << s))
            wait_bounded(smem_u32(&full[s]), (last_parity >> s) & 1, abort_flag, &g_device_status, kDrainLimitNs, false);
      } else if (!ok) {
        // The peer cannot observe its copies' completion (they signal the leader): after an
        // abort give copies in flight time to land before the final cluster barrier.
        const uint64_t t0 = global_ns();
        while (global_ns() - t0 < 100000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------- MMA issuer -------------
    if (lane == 0 && leader) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int it = cluster_id; it < num_items && ok; it += num_clusters, ++local) {
        const Item w = item_of(it, g);
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bounded(smem_u32(&tempty[acc]), acc_phase ^ 1, abort_flag, &g_device_status, kWaitLimitNs, true)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = w.kb0; kb < w.kb1; ++kb) {
          if (!mbar_try_wait(smem_u32(&full[stage]), phase) &&
              !wait_bounded(smem_u32(&full[stage]), phase, abort_flag, &g_device_status, kWaitLimitNs, true)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smA + stage * A_STAGE);
          const uint32_t b_base = smem_u32(smB + stage * B_STAGE);
#pragma unroll
          for (int j = 0; j < kRowBytes / MMA_K_BYTES; ++j) {
            const uint64_t ad =
                A_KMAJOR ? smem_desc(a_base + j * MMA_K_BYTES, 16, 8 * kRowBytes)
                         : smem_desc(a_base + j * MMA_K * kRowBytes, EPR * kRowBytes, 8 * kRowBytes);
            const uint64_t bd =
                B_KMAJOR ? smem_desc(b_base + j * MMA_K_BYTES, 16, 8 * kRowBytes)
                         : smem_desc(b_base + j * MMA_K * kRowBytes, EPR * kRowBytes, 8 * kRowBytes);
            umma<KIND, CG>(d_tmem, ad, bd, IDESC, (kb != w.kb0 || j != 0) ? 1u : 0u);
          }
          if constexpr (CG == 1) umma_commit<1>(smem_u32(&empty[stage]));
          else umma_commit_mc(smem_u32(&empty[stage]), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        if constexpr (CG == 1) umma_commit<1>(smem_u32(&tfull[acc]));
        else umma_commit_mc(smem_u32(&tfull[acc]), 0x3);
      }
      // Own MMAs complete before TMEM is released.
      umma_commit<CG>(smem_u32(drain));
      wait_bounded(smem_u32(drain), 0, abort_flag, &g_device_status, kDrainLimitNs, false);
    }
  } else {
    // ----------------------------------------------------------- epilogue ---------------
    // Warp w reads the TMEM lanes of quadrant (w % 4) and one half of the tile's columns.
    const int quad = warp & 3;  // TMEM lanes [32 * quad, 32 * quad + 32)
    const int half = (warp - 2) >> 2;
    const int row_in_tile = quad * 32 + lane;
    float alpha = 1.0f;
    if (g.a_scale_inv) alpha *= *g.a_scale_inv;
    if (g.b_scale_inv) alpha *= *g.b_scale_inv;
    const f32x2 alpha2 = f2s(alpha);
    const float out_scale = (g.d_dtype == TE_E4M3 && g.out_scale) ? *g.out_scale : 1.0f;
    if (blockIdx.x == 0 && threadIdx.x == 64 && g.out_scale_inv) *g.out_scale_inv = 1.0f / out_scale;
    const uint32_t tempty_leader0 = CG == 1 ? smem_u32(&tempty[0]) : map_to_rank(smem_u32(&tempty[0]), 0);
    const uint32_t tempty_leader1 = CG == 1 ? smem_u32(&tempty[1]) : map_to_rank(smem_u32(&tempty[1]), 0);
    const int64_t ldd = g.gated ? g.F : g.N;
    const bool round_h = g.h_dtype == TE_BF16;
    const int gact = gate_act(g.act);  // a gated pair's function of its gate half
    float amax = 0.0f;
    int local = 0;
    uint32_t epi_phase = 0;
    // All epilogue warps meet (bounded like every other wait).
    auto epi_sync = [&]() -> bool {
      mbar_arrive(smem_u32(epi_bar));
      const bool r = wait_bounded(smem_u32(epi_bar), epi_phase, abort_flag, &g_device_status, kWaitLimitNs, true);
      epi_phase ^= 1;
      return r;
    };
    for (int it = cluster_id; it < num_items; it += num_clusters, ++local) {
      const Item w = item_of(it, g);
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const uint32_t tb = smem_u32(&tfull[acc]);
      int ok = 1;
      if (lane == 0) ok = wait_bounded(tb, acc_phase, abort_flag, &g_device_status, kWaitLimitNs, true) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // The phase has completed; every lane observes it before touching TMEM.
      while (!mbar_try_wait(tb, acc_phase)) {
      }
      __syncwarp();
      tc_fence_after();
      const Tile tl = tile_of(w.tile, g.num_m, g.num_n, g.group_m, g.n_major);
      const int64_t row = (int64_t(tl.m) * CG + rank) * BM + row_in_tile;
      const bool row_ok = row < g.M;
      const uint32_t taddr = tmem_base + (uint32_t(quad * 32) << 16) + uint32_t(acc * BN);
      // A K chunk of a split tile: every chunk stores its raw accumulator; the one counted in
      // last adds the others' to its own in TMEM, in chunk order, and runs the epilogue.
      bool epilogue = true;
      if (w.chunk >= 0) {
        const int u = w.tile - g.full_tiles;
        float* slot0 = g.partials + (size_t(u) * g.split * CG + rank) * (BM * BN);
        float* mine = slot0 + size_t(w.chunk) * CG * (BM * BN);
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
          const int col = epilogue_column(k, half, g.gated);
          uint32_t r[32];
          tmem_ld32(taddr + col, r);
          tmem_ld_wait();
          store_partial(mine, col, row_in_tile, r);
        }
        __threadfence();
        if (!epi_sync()) break;
        if (warp == 2 && lane == 0) split_arrival[local & 1] = atom_add_acq_rel(g.flags + u * CG + rank, 1);
        if (!epi_sync()) break;
        epilogue = split_arrival[local & 1] == g.split - 1;
        if (epilogue) {
          __threadfence();
#pragma unroll 1
          for (int k = 0; k < 4; ++k) {  // the columns this warp's epilogue reads back
            const int col = epilogue_column(k, half, g.gated);
            uint32_t r[32];
            tmem_ld32(taddr + col, r);
            tmem_ld_wait();
            add_chunks<CG>(r, slot0, w.chunk, g.split, col, row_in_tile);
            tmem_st32(taddr + col, r);
          }
          tmem_st_wait();
        }
      }
      if (epilogue && !g.gated) {
        const int64_t n0 = int64_t(tl.n) * BN;
        constexpr int kChunks = BN / 32 / 2;  // per warp
#pragma unroll 1
        for (int c = half * kChunks; c < (half + 1) * kChunks; ++c) {
          const int64_t col0 = n0 + c * 32;
          if (col0 >= g.N) break;
          const int count = g.N - col0 >= 32 ? 32 : int(g.N - col0);
          uint32_t r[32];
          tmem_ld32(taddr + c * 32, r);
          f32x2 bz[16];  // the chunk's bias, loaded while the accumulator columns arrive
          load_bias_chunk(g.bias, g.bias_dtype, col0, count, bz);
          tmem_ld_wait();
          float v[32];
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            f32x2 x = fma2(f2(__uint_as_float(r[2 * p]), __uint_as_float(r[2 * p + 1])), alpha2, bz[p]);
            if (g.epilogue == EPI_BIAS_ACT && round_h) x = round_bf16_2(x);
            v[2 * p] = f2lo(x);
            v[2 * p + 1] = f2hi(x);
          }
          if (g.epilogue == EPI_BIAS_ACT) {
            if (g.saved_h && row_ok) store_seg(g.saved_h, row * g.N + col0, v, count, g.h_dtype, 1.0f);
            act_chunk(g.act, v);
          }
          if (row_ok) {
            if (g.amax_out) amax = chunk_amax(amax, v, count);
            store_seg(g.D, row * ldd + col0, v, count, g.d_dtype, out_scale);
          }
        }
      } else if (epilogue) {
        const int64_t n0 = int64_t(tl.n) * (BN / 2);
        constexpr int kChunks = BN / 64 / 2;  // per warp
#pragma unroll 1
        for (int c = half * kChunks; c < (half + 1) * kChunks; ++c) {
          const int64_t col0 = n0 + c * 32;
          if (col0 >= g.F) break;
          const int count = g.F - col0 >= 32 ? 32 : int(g.F - col0);
          uint32_t rg[32], rl[32];
          tmem_ld32(taddr + c * 32, rg);
          tmem_ld32(taddr + BN / 2 + c * 32, rl);
          f32x2 bg[16], bl[16];
          load_bias_chunk(g.bias, g.bias_dtype, col0, count, bg);
          load_bias_chunk(g.bias, g.bias_dtype, g.F + col0, count, bl);
          tmem_ld_wait();
          float vg[32], vl[32];
#pragma unroll
          for (int p = 0; p < 16; ++p) {
            f32x2 xg = fma2(f2(__uint_as_float(rg[2 * p]), __uint_as_float(rg[2 * p + 1])), alpha2, bg[p]);
            f32x2 xl = fma2(f2(__uint_as_float(rl[2 * p]), __uint_as_float(rl[2 * p + 1])), alpha2, bl[p]);
            if (round_h) {
              xg = round_bf16_2(xg);
              xl = round_bf16_2(xl);
            }
            vg[2 * p] = f2lo(xg);
            vg[2 * p + 1] = f2hi(xg);
            vl[2 * p] = f2lo(xl);
            vl[2 * p + 1] = f2hi(xl);
          }
          if (g.saved_h && row_ok) {
            store_seg(g.saved_h, row * g.N + col0, vg, count, g.h_dtype, 1.0f);
            store_seg(g.saved_h, row * g.N + g.F + col0, vl, count, g.h_dtype, 1.0f);
          }
          gated_chunk(gact, vg, vl);
          if (row_ok) {
            if (g.amax_out) amax = chunk_amax(amax, vg, count);
            store_seg(g.D, row * ldd + col0, vg, count, g.d_dtype, out_scale);
          }
        }
      }
      tc_fence_before();
      if constexpr (CG == 1) mbar_arrive(acc ? tempty_leader1 : tempty_leader0);
      else mbar_arrive_cluster(acc ? tempty_leader1 : tempty_leader0);
    }
    amax = warp_max(amax);
    if (lane == 0 && g.amax_out) atomic_max_nonneg(g.amax_out, amax);
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (CG == 2) cluster_sync();  // no MMA of the pair still writes this CTA's TMEM
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<CG>(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side -------------

template <int KIND, bool AK, bool BK, int CG>
te_status launch_t(GemmParams& prm, int grid, cudaStream_t s) {
  constexpr size_t smem = Cfg<CG>::kSmem;
  static PerDevice<bool> attr_set;
  bool ok = false;
  if (!attr_set.get(&ok, [](bool* v) {
        *v = cudaFuncSetAttribute(gemm_kernel<KIND, AK, BK, CG>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  int(smem)) == cudaSuccess;
        return *v;
      }))
    return TE_ERR_CUDA;
  // a programmatic dependent launch (the kernel waits for its predecessor after its setup),
  // in clusters of two CTAs for the SM-pair form
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CG;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = CG == 1 ? 1 : 2;
  if (cudaLaunchKernelEx(&cfg, gemm_kernel<KIND, AK, BK, CG>, prm) != cudaSuccess) return TE_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? TE_OK : TE_ERR_CUDA;
}

template <int KIND, int CG>
te_status launch_kind(GemmParams& prm, int grid, bool ak, bool bk, cudaStream_t s) {
  if (ak && bk) return launch_t<KIND, true, true, CG>(prm, grid, s);
  if (ak && !bk) return launch_t<KIND, true, false, CG>(prm, grid, s);
  if (!ak && bk) return launch_t<KIND, false, true, CG>(prm, grid, s);
  return launch_t<KIND, false, false, CG>(prm, grid, s);
}

// CTAs per MMA: pairs for bf16 / E4M3 problems taller than one tile.  TE_GEMM_CTA_GROUP=1 in
// the environment forces single-CTA tiles (a diagnostic switch between two complete paths).
int choose_cta_group(int kind, int64_t M) {
  static int forced = -1;
  if (forced < 0) {
    const char* e = getenv("TE_GEMM_CTA_GROUP");
    forced = (e && e[0] == '1') ? 1 : 0;
  }
  if (forced == 1 || kind == 2 || M <= BM) return 1;
  return 2;
}

// Tile grid of one GEMM.
struct Geometry {
  int kind, esize, cg, num_m, num_n, num_kb;
};

Geometry geometry(int ab_dtype, int64_t M, int64_t N, int64_t K, bool gated) {
  Geometry q;
  q.kind = ab_dtype == TE_BF16 ? 0 : ab_dtype == TE_E4M3 ? 1 : 2;
  q.esize = ab_dtype == TE_BF16 ? 2 : ab_dtype == TE_E4M3 ? 1 : 4;
  q.cg = choose_cta_group(q.kind, M);
  q.num_m = int(ceil_div(M, int64_t(BM) * q.cg));
  q.num_n = int(gated ? ceil_div(N / 2, BN / 2) : ceil_div(N, BN));
  q.num_kb = int(ceil_div(K, int64_t(kRowBytes / q.esize)));
  return q;
}

// K split of the tiles left over after the last whole wave.  A tile keeps its SM pair busy for
// about num_kb k-block times (about a third of a microsecond each, for every operand type).
// Splitting pays only while all chunks run at once, in one wave: spread over several waves, the
// chunks of one tile re-read their operands in different waves and lose more than they gain.
// Measured on GB300, storing a chunk's partial and summing the partials cost about 24 k-block
// times per chunk.  The plan takes the split that finishes the leftover tiles soonest, within
// the workspace given.  TE_GEMM_SPLIT_K=0 in the environment turns splitting off (a diagnostic
// switch between two complete paths).
constexpr int kSplitCostKb = 24;
constexpr int kMinChunkKb = 4;

struct SplitPlan {
  int64_t full_tiles = 0;
  int split = 1;
  int kb_chunk = 0;
  size_t partial_bytes = 0;
  size_t flag_bytes = 0;
};

bool split_enabled() {
  const char* e = getenv("TE_GEMM_SPLIT_K");
  return !(e && e[0] == '0');
}

SplitPlan plan_split(int64_t tiles, int64_t clusters, int num_kb, int cg, size_t budget) {
  SplitPlan best;
  best.full_tiles = tiles;
  best.kb_chunk = num_kb;
  if (clusters < 1 || tiles < 1) return best;
  const int64_t full = tiles / clusters * clusters;
  const int64_t rest = tiles - full;
  if (rest == 0) return best;
  int64_t best_cost = num_kb;  // unsplit: one round of whole tiles
  for (int sp : {2, 3, 4, 6, 8}) {
    const int kbc = (num_kb + sp - 1) / sp;
    if (kbc < kMinChunkKb || int64_t(sp - 1) * kbc >= num_kb) continue;  // every chunk non-empty
    if (rest * sp > clusters) break;  // more than one wave of chunks
    const int64_t cost = kbc + int64_t(kSplitCostKb) * sp;
    const size_t pb = size_t(rest) * sp * cg * BM * BN * sizeof(float);
    const size_t fb = (size_t(rest) * cg * sizeof(int) + 255) / 256 * 256;
    if (cost >= best_cost || pb + fb > budget) continue;
    best_cost = cost;
    best.full_tiles = full;
    best.split = sp;
    best.kb_chunk = kbc;
    best.partial_bytes = pb;
    best.flag_bytes = fb;
  }
  return best;
}

}  // namespace

int num_sms() {
  static PerDevice<int> cached;
  int n = 1;
  if (!cached.get(&n, [](int* v) {
        int dev = 0, count = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            count < 1)
          return false;
        *v = count;
        return true;
      }))
    return 1;
  return n;
}

int* device_status_ptr() {
  static PerDevice<int*> cached;
  int* p = nullptr;
  if (!cached.get(&p, [](int** v) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess || !addr) return false;
        *v = static_cast<int*>(addr);
        return true;
      }))
    return nullptr;
  return p;
}

te_status read_and_clear_device_status(int32_t* out) {
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return TE_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return TE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return TE_ERR_CUDA;
  if (out) *out = v;
  return TE_OK;
}

size_t gemm_split_workspace(int64_t M, int64_t N, int64_t K, int ab_dtype, int epilogue) {
  if (M <= 0 || N <= 0 || K <= 0) return 0;
  const Geometry q = geometry(ab_dtype, M, N, K, epilogue == EPI_BIAS_GATED);
  const SplitPlan sp = plan_split(int64_t(q.num_m) * q.num_n, num_sms() / q.cg, q.num_kb, q.cg, SIZE_MAX);
  return sp.partial_bytes + sp.flag_bytes;
}

te_status launch_gemm(const GemmArgs& a, cudaStream_t s) {
  if (a.M == 0 || a.N == 0) return TE_OK;
  const bool gated = a.epilogue == EPI_BIAS_GATED;
  const Geometry q = geometry(a.ab_dtype, a.M, a.N, a.K, gated);
  const int kind = q.kind;
  const int esize = q.esize;
  const uint32_t epr = uint32_t(kRowBytes / esize);
  const int cg = q.cg;
  GemmParams prm;
  memset(&prm, 0, sizeof(prm));
  // A: op(A) is [M, K]; each CTA loads 128 rows.
  bool ok = a.a_kmajor ? make_tmap_2d(&prm.tmA, a.A, a.ab_dtype, a.K, a.M, epr, BM, true)
                       : make_tmap_2d(&prm.tmA, a.A, a.ab_dtype, a.M, a.K, epr, epr, true);
  // B: op(B) is [K, N]; a K-major box holds the B columns one CTA loads at a time.
  const uint32_t b_rows = (gated || cg == 2) ? BN / 2 : BN;
  ok = ok && (a.b_kmajor ? make_tmap_2d(&prm.tmB, a.B, a.ab_dtype, a.K, a.N, epr, b_rows, true)
                         : make_tmap_2d(&prm.tmB, a.B, a.ab_dtype, a.N, a.K, epr, epr, true));
  if (!ok) return TE_ERR_CUDA;
  GemmDev& g = prm.g;
  g.M = a.M;
  g.N = a.N;
  g.K = a.K;
  g.gated = gated ? 1 : 0;
  g.F = gated ? a.N / 2 : 0;
  g.num_m = q.num_m;
  g.num_n = q.num_n;
  g.num_kb = q.num_kb;
  {
    const int64_t a_tile_bytes = int64_t(BM) * cg * a.K * esize;
    int64_t gm = kRasterL2Bytes / (a_tile_bytes > 0 ? a_tile_bytes : 1);
    if (gm < 4) gm = 4;
    g.group_m = int(gm < g.num_m ? gm : g.num_m);
    // B small enough to stay in L2 while A streams once (measured on the FP8 Llama GEMM2, B =
    // 58.7 MB: +3% against m-major groups, which read B about three times)
    const int64_t b_bytes = a.K * a.N * esize;
    g.n_major = (g.num_n > 1 && b_bytes <= kBResidentBytes) ? 1 : 0;
  }
  g.epilogue = a.epilogue;
  g.act = a.act;
  g.a_scale_inv = a.a_scale_inv;
  g.b_scale_inv = a.b_scale_inv;
  g.bias = a.bias;
  g.bias_dtype = a.bias_dtype;
  g.h_dtype = a.h_dtype;
  g.saved_h = a.saved_h;
  g.D = a.D;
  g.d_dtype = a.cast.out_dtype;
  g.out_scale = a.cast.scale;
  g.out_scale_inv = a.cast.scale_inv_out;
  g.amax_out = a.cast.amax_out;
  const int64_t tiles = int64_t(g.num_m) * g.num_n;
  const int64_t slots = num_sms() / cg;
  SplitPlan sp;
  sp.full_tiles = tiles;
  sp.kb_chunk = g.num_kb;
  if (a.split_ws && split_enabled()) sp = plan_split(tiles, slots, g.num_kb, cg, a.split_ws_bytes);
  g.full_tiles = int(sp.full_tiles);
  g.split = sp.split;
  g.kb_chunk = sp.kb_chunk;
  if (sp.split > 1) {
    g.partials = static_cast<float*>(a.split_ws);
    g.flags = reinterpret_cast<int*>(static_cast<char*>(a.split_ws) + sp.partial_bytes);
    if (cudaMemsetAsync(g.flags, 0, sp.flag_bytes, s) != cudaSuccess) return TE_ERR_CUDA;
  }
  const int64_t items = sp.full_tiles + (tiles - sp.full_tiles) * sp.split;
  const int grid = int(items < slots ? items : slots) * cg;
  ProfileScope prof(a.epilogue == EPI_BIAS ? TE_KERNEL_GEMM : TE_KERNEL_GEMM_ACT, s);
  if (cg == 1) {
    if (kind == 0) return launch_kind<0, 1>(prm, grid, a.a_kmajor, a.b_kmajor, s);
    if (kind == 1) return launch_kind<1, 1>(prm, grid, a.a_kmajor, a.b_kmajor, s);
    return launch_kind<2, 1>(prm, grid, a.a_kmajor, a.b_kmajor, s);
  }
  if (kind == 0) return launch_kind<0, 2>(prm, grid, a.a_kmajor, a.b_kmajor, s);
  return launch_kind<1, 2>(prm, grid, a.a_kmajor, a.b_kmajor, s);
}

}  // namespace te
