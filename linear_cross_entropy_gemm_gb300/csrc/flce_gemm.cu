// Instantiations and launchers of the persistent tcgen05 GEMMs.
#include <atomic>
#include <cstdlib>

#include <cuda_runtime.h>

#include "epilogues.cuh"
#include "flce_internal.h"

namespace flce {

template <class Epi>
static cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                          const typename Epi::Args& ea, int* dev_err, int grid, cudaStream_t st) {
  auto kernel = gemm_persistent<Epi>;
  // Setting the attribute is idempotent and cheap; doing it per launch keeps
  // the library free of per-device global state.
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmemBytes));
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, kSmemBytes, st>>>(a, b, g, ea, dev_err);
  return cudaGetLastError();
}

// Co-resident 2-CTA clusters of a cluster kernel on the current device,
// queried once per device and footprint (slot 0: the 256 x 256 pair kernel,
// whose instantiations share one footprint; slots 1 and 2: the wide pair
// kernel with 8 and 16 epilogue warps).
static int max_pair_clusters(const void* kernel, int slot, int threads, size_t smem) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[3][kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int v = cache[slot][dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&v, kernel, &cfg) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    return 0;
  }
  cache[slot][dev].store(v, std::memory_order_relaxed);
  return v;
}

template <class Epi>
static cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                               const typename Epi::Args& ea, int* dev_err, int sms,
                               cudaStream_t st) {
  auto kernel = gemm_persistent_pair<Epi>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kPairSmemBytes));
  if (e != cudaSuccess) return e;
  int clusters = max_pair_clusters(reinterpret_cast<const void*>(kernel), 0, kThreads,
                                   kPairSmemBytes);
  if (clusters <= 0) clusters = sms / 2;
  const int pair_tiles = ((g.tiles_m + 1) / 2) * g.tiles_n;
  if (clusters > pair_tiles) clusters = pair_tiles;
  kernel<<<2 * clusters, kThreads, kPairSmemBytes, st>>>(a, b, g, ea, dev_err);
  return cudaGetLastError();
}

template <class Epi, int kEW>
static cudaError_t launch_wide_warps(const CUtensorMap& a, const CUtensorMap& b,
                                     const GemmGeom& g, const typename Epi::Args& ea,
                                     int* dev_err, int sms, cudaStream_t st) {
  auto kernel = gemm_persistent_wide<Epi, kEW>;
  constexpr int threads = wide_threads(kEW);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kWideSmemBytes));
  if (e != cudaSuccess) return e;
  int clusters = max_pair_clusters(reinterpret_cast<const void*>(kernel), kEW == 16 ? 2 : 1,
                                   threads, kWideSmemBytes);
  if (clusters <= 0) clusters = sms / 2;
  const int wide_tiles = ((g.tiles_m + 1) / 2) * ((g.tiles_n + 1) / 2);
  if (clusters > wide_tiles) clusters = wide_tiles;
  kernel<<<2 * clusters, threads, kWideSmemBytes, st>>>(a, b, g, ea, dev_err);
  return cudaGetLastError();
}

// FLCE_WIDE_EPI_WARPS=8 runs every wide epilogue on 8 warps (an A/B switch;
// by default each epilogue's kWideWarps applies).
static bool wide_epi_warps_forced_8() {
  const char* e = std::getenv("FLCE_WIDE_EPI_WARPS");
  return e && std::atoi(e) == 8;
}

template <class Epi>
static cudaError_t launch_wide(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                               const typename Epi::Args& ea, int* dev_err, int sms,
                               cudaStream_t st) {
  if constexpr (Epi::kWideWarps == 16) {
    if (!wide_epi_warps_forced_8())
      return launch_wide_warps<Epi, 16>(a, b, g, ea, dev_err, sms, st);
  }
  return launch_wide_warps<Epi, 8>(a, b, g, ea, dev_err, sms, st);
}

template <class Epi>
static cudaError_t launch_any(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                              const GemmGeom& g, const typename Epi::Args& ea, int* dev_err,
                              int grid, cudaStream_t st) {
  switch (kind) {
    case kGemmWide: return launch_wide<Epi>(a, b, g, ea, dev_err, grid, st);
    case kGemmSingle: return launch<Epi>(a, b, g, ea, dev_err, grid, st);
    default: return launch_pair<Epi>(a, b, g, ea, dev_err, grid, st);  // kGemmAuto is resolved earlier
  }
}

template <bool KEEP>
static cudaError_t launch_fwd_lse_t(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                                    const GemmGeom& g, const FwdLseArgs& ea, bool has_bias,
                                    bool has_smooth, int* dev_err, int grid, cudaStream_t st) {
  if (has_bias)
    return has_smooth
               ? launch_any<FwdLseEpi<true, true, KEEP>>(kind, a, b, g, ea, dev_err, grid, st)
               : launch_any<FwdLseEpi<true, false, KEEP>>(kind, a, b, g, ea, dev_err, grid, st);
  return has_smooth
             ? launch_any<FwdLseEpi<false, true, KEEP>>(kind, a, b, g, ea, dev_err, grid, st)
             : launch_any<FwdLseEpi<false, false, KEEP>>(kind, a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_fwd_lse(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const FwdLseArgs& ea, bool has_bias,
                           bool has_smooth, bool keep, int* dev_err, int grid, cudaStream_t st) {
  return keep ? launch_fwd_lse_t<true>(kind, a, b, g, ea, has_bias, has_smooth, dev_err, grid, st)
              : launch_fwd_lse_t<false>(kind, a, b, g, ea, has_bias, has_smooth, dev_err, grid,
                                        st);
}

cudaError_t launch_dlogits(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const DlogitsArgs& ea, bool has_bias, int* dev_err,
                           int grid, cudaStream_t st) {
  return has_bias ? launch_any<DlogitsEpi<true>>(kind, a, b, g, ea, dev_err, grid, st)
                  : launch_any<DlogitsEpi<false>>(kind, a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dw(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DwArgs& ea, int* dev_err, int grid, cudaStream_t st) {
  return launch_any<DwEpi>(kind, a, b, g, ea, dev_err, grid, st);
}

// dx has few output tiles (N/256 x H/256) and a long K: 256 x 512 tiles would
// leave most of the GPU idle in the last wave, so the wide form runs it as pairs.
cudaError_t launch_dx(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DxArgs& ea, int* dev_err, int grid, cudaStream_t st) {
  return launch_any<DxEpi>(kind == kGemmWide ? kGemmPair : kind, a, b, g, ea, dev_err, grid, st);
}

}  // namespace flce
