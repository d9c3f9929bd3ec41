// Instantiations and launchers of the persistent tcgen05 GEMMs.
#include <atomic>

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

// Co-resident 2-CTA clusters of gemm_persistent_pair on the current device,
// queried once per device (all instantiations share the same footprint).
static int max_pair_clusters(const void* kernel) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kPairSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&v, kernel, &cfg) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    return 0;
  }
  cache[dev].store(v, std::memory_order_relaxed);
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
  int clusters = max_pair_clusters(reinterpret_cast<const void*>(kernel));
  if (clusters <= 0) clusters = sms / 2;
  const int pair_tiles = ((g.tiles_m + 1) / 2) * g.tiles_n;
  if (clusters > pair_tiles) clusters = pair_tiles;
  kernel<<<2 * clusters, kThreads, kPairSmemBytes, st>>>(a, b, g, ea, dev_err);
  return cudaGetLastError();
}

template <class Epi>
static cudaError_t launch_any(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                              const GemmGeom& g, const typename Epi::Args& ea, int* dev_err,
                              int grid, cudaStream_t st) {
  return pair ? launch_pair<Epi>(a, b, g, ea, dev_err, grid, st)
              : launch<Epi>(a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_fwd_lse(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const FwdLseArgs& ea, bool has_bias,
                           bool has_smooth, int* dev_err, int grid, cudaStream_t st) {
  if (has_bias)
    return has_smooth ? launch_any<FwdLseEpi<true, true>>(pair, a, b, g, ea, dev_err, grid, st)
                      : launch_any<FwdLseEpi<true, false>>(pair, a, b, g, ea, dev_err, grid, st);
  return has_smooth ? launch_any<FwdLseEpi<false, true>>(pair, a, b, g, ea, dev_err, grid, st)
                    : launch_any<FwdLseEpi<false, false>>(pair, a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_fwd_store(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                             const GemmGeom& g, const FwdStoreArgs& ea, bool has_bias,
                             bool has_smooth, int* dev_err, int grid, cudaStream_t st) {
  if (has_bias)
    return has_smooth ? launch_any<FwdStoreEpi<true, true>>(pair, a, b, g, ea, dev_err, grid, st)
                      : launch_any<FwdStoreEpi<true, false>>(pair, a, b, g, ea, dev_err, grid, st);
  return has_smooth ? launch_any<FwdStoreEpi<false, true>>(pair, a, b, g, ea, dev_err, grid, st)
                    : launch_any<FwdStoreEpi<false, false>>(pair, a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dlogits(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const DlogitsArgs& ea, bool has_bias, int* dev_err,
                           int grid, cudaStream_t st) {
  return has_bias ? launch_any<DlogitsEpi<true>>(pair, a, b, g, ea, dev_err, grid, st)
                  : launch_any<DlogitsEpi<false>>(pair, a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dw(bool pair, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DwArgs& ea, int* dev_err, int grid, cudaStream_t st) {
  return launch_any<DwEpi>(pair, a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dx(bool pair, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DxArgs& ea, int* dev_err, int grid, cudaStream_t st) {
  return launch_any<DxEpi>(pair, a, b, g, ea, dev_err, grid, st);
}

}  // namespace flce
