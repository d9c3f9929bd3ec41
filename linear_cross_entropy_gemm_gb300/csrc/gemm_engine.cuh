// Persistent, warp-specialised tcgen05 GEMM engine shared by every
// contraction of the fused linear cross-entropy (FLCE) path.
//
//   D[M, N] = A[M, K] * B[N, K]^T   (bf16 or fp16 in, fp32 accumulate in TMEM)
//
// One CTA per SM (192 threads):
//   warp 0      TMA producer: a kStages-deep ring of (A, B) K-slices in smem
//   warp 1      MMA issuer (one thread): tcgen05.mma 128x256x16 into one of
//               two TMEM accumulators (2 x 256 fp32 columns = all 512)
//   warps 2..5  epilogue: 128 threads, thread i owns accumulator row (TMEM
//               lane) i; drains tile t while the MMAs of tile t+1 run
// The tile loop is persistent (tile = blockIdx.x + j * gridDim.x), in an
// order chosen per problem so the operand shared by concurrent CTAs stays in L2.
// Two cluster forms follow the single-CTA one: gemm_persistent_pair (two CTAs,
// cta_group::2, one 256 x 256 tile) and gemm_persistent_wide (two CTAs, one
// 256 x 512 tile as two MMAs per K step sharing A, 8 or 16 epilogue warps).
//
// Operands are 128-byte-swizzled 16-bit tiles loaded by TMA, either K-major
// (rows of 64 contiguous K elements) or MN-major (rows of 64 contiguous M/N
// elements, one per K index); the tcgen05 instruction descriptor's transpose
// bits select the form, so dW = dL^T x and dx = dL W need no transposed copies.
#pragma once
#include <cstdint>
#include <cuda.h>

#include "sm103_primitives.cuh"

namespace flce {

constexpr int kBM = 128;      // accumulator rows (TMEM lanes)
constexpr int kBN = 256;      // accumulator columns per buffer
constexpr int kBK = 64;       // K elements per pipeline stage (one 128-B swizzle row)
constexpr int kUmmaK = 16;    // K per tcgen05.mma (kind::f16)
constexpr int kStages = 4;
constexpr int kAStageBytes = kBM * kBK * 2;   // 16 KiB
constexpr int kBStageBytes = kBN * kBK * 2;   // 32 KiB
constexpr int kThreads = 192;
constexpr int kEpiThreads = 128;
constexpr int kTmemCols = 2 * kBN;
constexpr int kMnBoxBytes = 64 * kBK * 2;     // one 64 (MN) x 64 (K) MN-major box
constexpr int kBarrierBytes = 256;
// Per epilogue warp: a staging buffer through which the epilogues transpose
// 32 x 32 blocks for coalesced global stores.
constexpr int kStageBytes = 4096;
constexpr size_t kSmemBytes = 1024 +
                              static_cast<size_t>(kStages) * (kAStageBytes + kBStageBytes) +
                              4 * kStageBytes + kBarrierBytes;

struct GemmGeom {
  int M, N, K;
  int tiles_m, tiles_n, k_blocks;
  int a_mn_off, a_k_off;  // added to the A / B load coordinates
  int b_mn_off, b_k_off;
  int raster_m_inner;     // 1: consecutive tiles advance along M first
  int band_m;             // >0: bands of band_m M-tiles; inside a band M inner, N outer
  int band_n;             // >0: bands of band_n N-tiles; inside a band N inner, M outer
  int ab_fp16;            // operands are fp16 (else bf16)
};

// The 32-column chunks of a 128 x 256 accumulator sub-tile that one epilogue
// warp drains. A warp takes all eight, or (in the 256 x 512 kernel with 16
// epilogue warps) one half of them while a partner warp of the same TMEM lane
// quarter takes the other; an epilogue whose row results span the sub-tile
// then combines them: the second warp publishes its 32 rows' results in xchg
// (its own staging buffer) and arrives on xbar, the first waits (bounded),
// reads them, arrives on xfree and merges. The second warp waits (bounded) on
// xfree before it touches its staging buffer again in the next sub-tile it
// hands off, so the hand-off never depends on how far ahead of its partner the
// kernel's accumulator scheme lets it run.
struct EpiSlice {
  int c_lo, c_hi;            // chunks [c_lo, c_hi) of the sub-tile's kBN / 32
  int sub;                   // -1: the whole sub-tile; 0 / 1: first / second half
  uint64_t* xbar;            // sub >= 0: "published" barrier of the pair (32 arrivals)
  uint64_t* xfree;           // sub >= 0: "read" barrier of the pair (32 arrivals)
  float4* xchg;              // sub >= 0: 32 slots, one per row, written by sub 1
  uint32_t xph;              // parity of xbar's phase for this sub-tile
  int xcount;                // hand-offs completed before this sub-tile
  volatile int* abort_flag;  // the CTA's abort flag (for the bounded wait)
  int* dev_err;
};

__device__ __forceinline__ EpiSlice whole_slice() {
  EpiSlice sl;
  sl.c_lo = 0;
  sl.c_hi = kBN / 32;
  sl.sub = -1;
  sl.xbar = nullptr;
  sl.xfree = nullptr;
  sl.xchg = nullptr;
  sl.xph = 0;
  sl.xcount = 0;
  sl.abort_flag = nullptr;
  sl.dev_err = nullptr;
  return sl;
}

__device__ __forceinline__ void tile_coords(const GemmGeom& g, int t, int& tm, int& tn) {
  if (g.band_m > 0) {
    // A band of band_m M-tiles sweeps every N-tile: its A rows stay in L2 while
    // the B operand streams; B is read once per band.
    const int per = g.band_m * g.tiles_n;
    const int b = t / per;
    const int r = t - b * per;
    const int height = min(g.band_m, g.tiles_m - b * g.band_m);
    tn = r / height;
    tm = b * g.band_m + (r - tn * height);
  } else if (g.band_n > 0) {
    // A band of band_n N-tiles sweeps every M-tile: its B columns stay in L2.
    const int per = g.band_n * g.tiles_m;
    const int b = t / per;
    const int r = t - b * per;
    const int width = min(g.band_n, g.tiles_n - b * g.band_n);
    tm = r / width;
    tn = b * g.band_n + (r - tm * width);
  } else if (g.raster_m_inner) {
    tm = t % g.tiles_m;
    tn = t / g.tiles_m;
  } else {
    tn = t % g.tiles_n;
    tm = t / g.tiles_n;
  }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > kWaitCycles) return;
  }
}

template <class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_persistent(const __grid_constant__ CUtensorMap mapA,
                    const __grid_constant__ CUtensorMap mapB, const GemmGeom g,
                    const __grid_constant__ typename Epi::Args ea, int* dev_err) {
  constexpr bool kAMN = Epi::kAMN;
  constexpr bool kBMN = Epi::kBMN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kAStageBytes;
  uint8_t* stage = sB + kStages * kBStageBytes;  // 4 epilogue warps x kStageBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + 4 * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done_bar = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kEpiThreads);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_tiles = g.tiles_m * g.tiles_n;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------ TMA producer
      const uint64_t pol_a = l2_policy_evict_normal(), pol_b = pol_a;
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        int tm, tn;
        tile_coords(g, t, tm, tn);
        const int m0 = tm * kBM, n0 = tn * kBN;
        bool ok = true;
        for (int kb = 0; kb < g.k_blocks; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], kAStageBytes + kBStageBytes);
          uint8_t* a = sA + s * kAStageBytes;
          uint8_t* b = sB + s * kBStageBytes;
          const int k0 = kb * kBK;
          if constexpr (!kAMN) {
            tma_load_2d(a, &mapA, &full[s], k0 + g.a_k_off, m0 + g.a_mn_off, pol_a);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j)
              tma_load_2d(a + j * kMnBoxBytes, &mapA, &full[s], m0 + g.a_mn_off + j * 64,
                          k0 + g.a_k_off, pol_a);
          }
          if constexpr (!kBMN) {
            tma_load_2d(b, &mapB, &full[s], k0 + g.b_k_off, n0 + g.b_mn_off, pol_b);
          } else {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              tma_load_2d(b + j * kMnBoxBytes, &mapB, &full[s], n0 + g.b_mn_off + j * 64,
                          k0 + g.b_k_off, pol_b);
          }
          ++issued;
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
      }
      // Drain: the last load issued into each stage must land before exit.
      for (long long i = (issued > kStages ? issued - kStages : 0); i < issued; ++i)
        mbar_drain(&full[i % kStages], static_cast<uint32_t>((i / kStages) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_f16kind_f32(kBM, kBN, kAMN, kBMN, g.ab_fp16 != 0);
      int s = 0;
      uint32_t ph = 0;
      int acc = 0;
      uint32_t aph = 0;
      for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
        if (!mbar_wait(&tempty[acc], aph ^ 1, abort_flag, dev_err)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < g.k_blocks; ++kb) {
          if (!mbar_wait(&full[s], ph, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(sA + s * kAStageBytes);
          const uint32_t b_addr = smem_u32(sB + s * kBStageBytes);
#pragma unroll
          for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
            const uint64_t ad = kAMN ? smem_desc_sw128(a_addr + kk * (kUmmaK * 128), kMnBoxBytes, 1024)
                                     : smem_desc_sw128(a_addr + kk * (kUmmaK * 2), 16, 1024);
            const uint64_t bd = kBMN ? smem_desc_sw128(b_addr + kk * (kUmmaK * 128), kMnBoxBytes, 1024)
                                     : smem_desc_sw128(b_addr + kk * (kUmmaK * 2), 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[s]);
          if (++s == kStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) aph ^= 1;
      }
      // Every MMA issued above must finish before TMEM is released.
      umma_commit(done_bar);
      mbar_drain(done_bar, 0);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int quad = warp & 3;  // TMEM lane quadrant this warp may access
    const int row_in_tile = quad * 32 + lane;
    const EpiSlice sl = whole_slice();
    int acc = 0;
    uint32_t aph = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
      int tm, tn;
      tile_coords(g, t, tm, tn);
      if (!mbar_wait(&tfull[acc], aph, abort_flag, dev_err)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      Epi::tile(ea, g, tm, tn, row_in_tile, lane, quad, taddr, stage + (warp - 2) * kStageBytes,
                sl);
      tc_fence_before();
      tmem_release_arrive(&tempty[acc]);
      acc ^= 1;
      if (acc == 0) aph ^= 1;
    }
    if (lane == 0) bulk_wait_group0();  // this warp's epilogue stores have completed
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

// ===========================================================================
// CTA-pair variant (cluster of 2, tcgen05 cta_group::2): one 256 x 256 tile
// per pair. CTA r loads rows [128 r, 128 r + 128) of the tile's A slice and of
// its B slice (16 KiB + 16 KiB per stage), so each SM streams a third less
// from L2 and writes a third less into shared memory than the single-CTA
// 128 x 256 tile. The even CTA issues the MMAs for both; each CTA's TMEM holds
// its 128 accumulator rows x 256 columns and its own 4 epilogue warps drain it.
//   full[s]   (even CTA) : both CTAs' TMA bytes of stage s
//   empty[s]  (each CTA) : pair MMA commit, multicast to both CTAs
//   tfull[a]  (each CTA) : pair MMA commit after a tile's last K step
//   tempty[a] (even CTA) : 256 epilogue arrivals, 128 from each CTA
constexpr int kPairStages = 6;
constexpr int kPairAStageBytes = kBM * kBK * 2;         // 16 KiB
constexpr int kPairBStageBytes = (kBN / 2) * kBK * 2;   // 16 KiB
constexpr size_t kPairSmemBytes =
    1024 + static_cast<size_t>(kPairStages) * (kPairAStageBytes + kPairBStageBytes) +
    4 * kStageBytes + kBarrierBytes;

template <class Epi>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_persistent_pair(const __grid_constant__ CUtensorMap mapA,
                         const __grid_constant__ CUtensorMap mapB, const GemmGeom g,
                         const __grid_constant__ typename Epi::Args ea, int* dev_err) {
  constexpr bool kAMN = Epi::kAMN;
  constexpr bool kBMN = Epi::kBMN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kPairStages * kPairAStageBytes;
  uint8_t* stage = sB + kPairStages * kPairBStageBytes;  // 4 epilogue warps x kStageBytes
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + 4 * kStageBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kPairStages;
  uint64_t* tfull = bars + 2 * kPairStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* done_bar = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 2 * kEpiThreads);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Pair tiles: 256 rows of M (two 128-row halves) x 256 columns of N.
  GemmGeom pg = g;
  pg.tiles_m = (g.tiles_m + 1) / 2;
  const int num_tiles = pg.tiles_m * pg.tiles_n;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer (both CTAs)
      const uint64_t pol_a = l2_policy_evict_normal(), pol_b = pol_a;
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (int t = cluster; t < num_tiles; t += nclusters) {
        int tm2, tn;
        tile_coords(pg, t, tm2, tn);
        const int m0 = tm2 * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int n0 = tn * kBN + static_cast<int>(rank) * (kBN / 2);
        bool ok = true;
        for (int kb = 0; kb < g.k_blocks; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          if (leader)
            mbar_arrive_expect_tx(&full[s], 2 * (kPairAStageBytes + kPairBStageBytes));
          const uint32_t fb = full0 + static_cast<uint32_t>(s) * 8u;
          uint8_t* a = sA + s * kPairAStageBytes;
          uint8_t* b = sB + s * kPairBStageBytes;
          const int k0 = kb * kBK;
          if constexpr (!kAMN) {
            tma_load_2d_pair(a, &mapA, fb, k0 + g.a_k_off, m0 + g.a_mn_off, pol_a);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j)
              tma_load_2d_pair(a + j * kMnBoxBytes, &mapA, fb, m0 + g.a_mn_off + j * 64,
                               k0 + g.a_k_off, pol_a);
          }
          if constexpr (!kBMN) {
            tma_load_2d_pair(b, &mapB, fb, k0 + g.b_k_off, n0 + g.b_mn_off, pol_b);
          } else {
#pragma unroll
            for (int j = 0; j < (kBN / 2) / 64; ++j)
              tma_load_2d_pair(b + j * kMnBoxBytes, &mapB, fb, n0 + g.b_mn_off + j * 64,
                               k0 + g.b_k_off, pol_b);
          }
          ++issued;
          if (++s == kPairStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
      }
      // Drain: a stage's loads have landed once the pair MMA that read it committed.
      for (long long i = (issued > kPairStages ? issued - kPairStages : 0); i < issued; ++i)
        mbar_drain(&empty[i % kPairStages], static_cast<uint32_t>((i / kPairStages) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // ------------------------------------------- MMA issuer (even CTA)
        const uint32_t idesc = idesc_f16kind_f32(2 * kBM, kBN, kAMN, kBMN, g.ab_fp16 != 0);
        int s = 0;
        uint32_t ph = 0;
        int acc = 0;
        uint32_t aph = 0;
        for (int t = cluster; t < num_tiles; t += nclusters) {
          if (!mbar_wait(&tempty[acc], aph ^ 1, abort_flag, dev_err)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kBN);
          bool ok = true;
          for (int kb = 0; kb < g.k_blocks; ++kb) {
            if (!mbar_wait(&full[s], ph, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + s * kPairAStageBytes);
            const uint32_t b_addr = smem_u32(sB + s * kPairBStageBytes);
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
              const uint64_t ad =
                  kAMN ? smem_desc_sw128(a_addr + kk * (kUmmaK * 128), kMnBoxBytes, 1024)
                       : smem_desc_sw128(a_addr + kk * (kUmmaK * 2), 16, 1024);
              const uint64_t bd =
                  kBMN ? smem_desc_sw128(b_addr + kk * (kUmmaK * 128), kMnBoxBytes, 1024)
                       : smem_desc_sw128(b_addr + kk * (kUmmaK * 2), 16, 1024);
              umma_bf16_pair(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
            }
            umma_commit_pair(&empty[s], 0x3);
            if (++s == kPairStages) {
              s = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
          umma_commit_pair(&tfull[acc], 0x3);
          acc ^= 1;
          if (acc == 0) aph ^= 1;
        }
        umma_commit_pair(done_bar, 0x3);
      }
      // Both CTAs: every pair MMA must finish before TMEM is released.
      mbar_drain(done_bar, 0);
    }
  } else {
    // ---------------------------------------------------- epilogue (both CTAs)
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    const EpiSlice sl = whole_slice();
    const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
    int acc = 0;
    uint32_t aph = 0;
    for (int t = cluster; t < num_tiles; t += nclusters) {
      int tm2, tn;
      tile_coords(pg, t, tm2, tn);
      if (!mbar_wait(&tfull[acc], aph, abort_flag, dev_err)) break;
      tc_fence_after();
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + static_cast<uint32_t>(acc * kBN);
      Epi::tile(ea, g, tm2 * 2 + static_cast<int>(rank), tn, row_in_tile, lane, quad, taddr,
                stage + (warp - 2) * kStageBytes, sl);
      tc_fence_before();
      tmem_release_arrive_cluster(tempty0 + static_cast<uint32_t>(acc) * 8u);
      acc ^= 1;
      if (acc == 0) aph ^= 1;
    }
    if (lane == 0) bulk_wait_group0();  // this warp's epilogue stores have completed
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

// ---------------------------------------------------------------------------
// Wide CTA pair: the two CTAs of a cluster compute one 256 x 512 tile as two
// cta_group::2 MMAs per K step (M=256, N=256 each) that share the A operand.
// Per stage each CTA loads its 128 rows of A (16 KiB) and two 128-row slices of
// B, one per N half (2 x 16 KiB): 768 operand rows per 2*256*512 flops against
// 512 per 2*256*256 for the 256 x 256 pair tile, a quarter fewer bytes moved
// from L2 into shared memory per flop. The 128 x 512 fp32 accumulator fills
// all 512 TMEM columns, so there is one accumulator: a tile's epilogue does not
// overlap the next tile's MMAs (the producer keeps prefetching meanwhile).
// The epilogue warps drain the two 256-column halves at the same time; each
// half is a 128 x 256 sub-tile for the same epilogues as the other forms.
// kEW = 8 gives each warp a whole sub-tile's rows of one TMEM lane quarter;
// kEW = 16 splits each sub-tile's columns between two warps of the same lane
// quarter (4 epilogue warps per SM sub-partition instead of 2: the drain is
// latency-bound, and it is exposed, since the accumulator fills TMEM).
//   full[s]  (even CTA) : both CTAs' TMA bytes of stage s
//   empty[s] (each CTA) : pair MMA commit, multicast to both CTAs
//   tfull    (each CTA) : pair MMA commit after a tile's last K step
//   tempty   (even CTA) : 2 x 32 kEW epilogue arrivals, one per epilogue thread
//   xbar[8]  (each CTA) : kEW = 16 only; a column-split warp pair's hand-off
//   xfree[8] (each CTA) : kEW = 16 only; the hand-off has been read
constexpr int kWideStages = 4;
constexpr int kWideBHalfBytes = (kBN / 2) * kBK * 2;           // 16 KiB
constexpr int kWideBStageBytes = 2 * kWideBHalfBytes;          // 32 KiB
constexpr int kWideStageRegion = 8 * kStageBytes;  // shared by the epilogue warps
constexpr size_t kWideSmemBytes =
    1024 + static_cast<size_t>(kWideStages) * (kPairAStageBytes + kWideBStageBytes) +
    kWideStageRegion + kBarrierBytes;
constexpr int wide_threads(int epi_warps) { return 64 + 32 * epi_warps; }

template <class Epi, int kEW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(wide_threads(kEW), 1)
    gemm_persistent_wide(const __grid_constant__ CUtensorMap mapA,
                         const __grid_constant__ CUtensorMap mapB, const GemmGeom g,
                         const __grid_constant__ typename Epi::Args ea, int* dev_err) {
  constexpr bool kAMN = Epi::kAMN;
  constexpr bool kBMN = Epi::kBMN;
  static_assert(kEW == 8 || kEW == 16, "8 or 16 epilogue warps");
  constexpr int kWarpStage = kWideStageRegion / kEW;  // staging bytes per epilogue warp
  static_assert(Epi::kStageNeed <= kWarpStage, "epilogue staging does not fit");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kWideStages * kPairAStageBytes;
  uint8_t* stage = sB + kWideStages * kWideBStageBytes;  // kEW epilogue warps x kWarpStage
  uint64_t* bars = reinterpret_cast<uint64_t*>(stage + kWideStageRegion);
  uint64_t* full = bars;
  uint64_t* empty = bars + kWideStages;
  uint64_t* tfull = bars + 2 * kWideStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* done_bar = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* xbar = done_bar + 2;  // [2 halves x 4 lane quarters], kEW = 16
  uint64_t* xfree = xbar + 8;     // [2 halves x 4 lane quarters], kEW = 16

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = blockIdx.x >> 1;
  const int nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWideStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * 32 * kEW);
    mbar_init(done_bar, 1);
    if constexpr (kEW == 16)
      for (int i = 0; i < 8; ++i) {
        mbar_init(&xbar[i], 32);
        mbar_init(&xfree[i], 32);
      }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Wide tiles: 256 rows of M (two 128-row halves, one per CTA) x 512 columns
  // of N (two 256-column halves, one per MMA). g's tile counts are in 128-row
  // and 256-column units; the raster runs over wide tiles.
  GemmGeom pg = g;
  pg.tiles_m = (g.tiles_m + 1) / 2;
  pg.tiles_n = (g.tiles_n + 1) / 2;
  const int num_tiles = pg.tiles_m * pg.tiles_n;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------- TMA producer (both CTAs)
      const uint64_t pol = l2_policy_evict_normal();
      const uint32_t full0 = mapa_shared(smem_u32(&full[0]), 0);
      int s = 0;
      uint32_t ph = 0;
      long long issued = 0;
      for (int t = cluster; t < num_tiles; t += nclusters) {
        int tm2, tn2;
        tile_coords(pg, t, tm2, tn2);
        const int m0 = tm2 * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int n0 = tn2 * (2 * kBN) + static_cast<int>(rank) * (kBN / 2);
        bool ok = true;
        for (int kb = 0; kb < g.k_blocks; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, abort_flag, dev_err)) {
            ok = false;
            break;
          }
          if (leader)
            mbar_arrive_expect_tx(&full[s], 2 * (kPairAStageBytes + kWideBStageBytes));
          const uint32_t fb = full0 + static_cast<uint32_t>(s) * 8u;
          uint8_t* a = sA + s * kPairAStageBytes;
          uint8_t* b = sB + s * kWideBStageBytes;
          const int k0 = kb * kBK;
          if constexpr (!kAMN) {
            tma_load_2d_pair(a, &mapA, fb, k0 + g.a_k_off, m0 + g.a_mn_off, pol);
          } else {
#pragma unroll
            for (int j = 0; j < kBM / 64; ++j)
              tma_load_2d_pair(a + j * kMnBoxBytes, &mapA, fb, m0 + g.a_mn_off + j * 64,
                               k0 + g.a_k_off, pol);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint8_t* bh = b + h * kWideBHalfBytes;
            const int nh = n0 + h * kBN + g.b_mn_off;
            if constexpr (!kBMN) {
              tma_load_2d_pair(bh, &mapB, fb, k0 + g.b_k_off, nh, pol);
            } else {
#pragma unroll
              for (int j = 0; j < (kBN / 2) / 64; ++j)
                tma_load_2d_pair(bh + j * kMnBoxBytes, &mapB, fb, nh + j * 64, k0 + g.b_k_off,
                                 pol);
            }
          }
          ++issued;
          if (++s == kWideStages) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
      }
      // Drain: a stage's loads have landed once the pair MMA that read it committed.
      for (long long i = (issued > kWideStages ? issued - kWideStages : 0); i < issued; ++i)
        mbar_drain(&empty[i % kWideStages], static_cast<uint32_t>((i / kWideStages) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // ------------------------------------------- MMA issuer (even CTA)
        const uint32_t idesc = idesc_f16kind_f32(2 * kBM, kBN, kAMN, kBMN, g.ab_fp16 != 0);
        int s = 0;
        uint32_t ph = 0;
        uint32_t aph = 0;
        for (int t = cluster; t < num_tiles; t += nclusters) {
          if (!mbar_wait(tempty, aph ^ 1, abort_flag, dev_err)) break;
          tc_fence_after();
          bool ok = true;
          for (int kb = 0; kb < g.k_blocks; ++kb) {
            if (!mbar_wait(&full[s], ph, abort_flag, dev_err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + s * kPairAStageBytes);
            const uint32_t b_addr = smem_u32(sB + s * kWideBStageBytes);
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
              const uint64_t ad =
                  kAMN ? smem_desc_sw128(a_addr + kk * (kUmmaK * 128), kMnBoxBytes, 1024)
                       : smem_desc_sw128(a_addr + kk * (kUmmaK * 2), 16, 1024);
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                const uint32_t bh = b_addr + static_cast<uint32_t>(h * kWideBHalfBytes);
                const uint64_t bd =
                    kBMN ? smem_desc_sw128(bh + kk * (kUmmaK * 128), kMnBoxBytes, 1024)
                         : smem_desc_sw128(bh + kk * (kUmmaK * 2), 16, 1024);
                umma_bf16_pair(tmem_base + static_cast<uint32_t>(h * kBN), ad, bd, idesc,
                               (kb | kk) != 0 ? 1u : 0u);
              }
            }
            umma_commit_pair(&empty[s], 0x3);
            if (++s == kWideStages) {
              s = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
          umma_commit_pair(tfull, 0x3);
          aph ^= 1;
        }
        umma_commit_pair(done_bar, 0x3);
      }
      // Both CTAs: every pair MMA must finish before TMEM is released.
      mbar_drain(done_bar, 0);
    }
  } else {
    // ----------------------------------------- epilogue (both CTAs, kEW warps)
    // Epilogue warp e = warp - 2 takes column slice e / 4 (kEW / 4 slices of
    // 512 / (kEW / 4) columns: N half, then the sub-tile's first or second 128
    // columns when kEW = 16) and reads TMEM lanes 32 (w % 4) .. 32 (w % 4) + 31.
    // A column-split pair is warps e and e + 4: same lane quarter, same SM
    // sub-partition; the second warp's staging buffer holds the hand-off.
    constexpr int kPerHalf = kEW / 8;  // warps per (lane quarter, N half)
    constexpr int kChunks = (kBN / 32) / kPerHalf;
    const int e = warp - 2;
    const int cs = e >> 2;
    const int half = cs / kPerHalf;
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    uint8_t* my_stage = stage + e * kWarpStage;
    EpiSlice sl;
    sl.sub = kPerHalf == 1 ? -1 : cs % kPerHalf;
    sl.c_lo = (sl.sub < 0 ? 0 : sl.sub) * kChunks;
    sl.c_hi = sl.c_lo + kChunks;
    sl.xbar = &xbar[half * 4 + quad];
    sl.xfree = &xfree[half * 4 + quad];
    sl.xchg = reinterpret_cast<float4*>(sl.sub == 0 ? my_stage + 4 * kWarpStage : my_stage);
    sl.xph = 0;
    sl.xcount = 0;
    sl.abort_flag = abort_flag;
    sl.dev_err = dev_err;
    const uint32_t tempty0 = mapa_shared(smem_u32(tempty), 0);
    uint32_t aph = 0;
    for (int t = cluster; t < num_tiles; t += nclusters) {
      int tm2, tn2;
      tile_coords(pg, t, tm2, tn2);
      if (!mbar_wait(tfull, aph, abort_flag, dev_err)) break;
      tc_fence_after();
      // The last wide tile's second half can lie wholly past N: no sub-tile.
      const int tn = tn2 * 2 + half;
      if (tn < g.tiles_n) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                               static_cast<uint32_t>(half * kBN);
        Epi::tile(ea, g, tm2 * 2 + static_cast<int>(rank), tn, row_in_tile, lane, quad, taddr,
                  my_stage, sl);
        sl.xph ^= 1;
        ++sl.xcount;
      }
      tc_fence_before();
      tmem_release_arrive_cluster(tempty0);
      aph ^= 1;
    }
    if (lane == 0) bulk_wait_group0();  // this warp's epilogue stores have completed
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, kTmemCols);
}

static_assert(kSmemBytes <= 232448 && kPairSmemBytes <= 232448 && kWideSmemBytes <= 232448,
              "dynamic shared memory above the 227 KiB a CTA may use");

}  // namespace flce
