// Instantiations and launchers of the persistent tcgen05 GEMMs.
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

cudaError_t launch_fwd_lse(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                           const FwdLseArgs& ea, bool has_bias, bool has_smooth, int* dev_err,
                           int grid, cudaStream_t st) {
  if (has_bias)
    return has_smooth ? launch<FwdLseEpi<true, true>>(a, b, g, ea, dev_err, grid, st)
                      : launch<FwdLseEpi<true, false>>(a, b, g, ea, dev_err, grid, st);
  return has_smooth ? launch<FwdLseEpi<false, true>>(a, b, g, ea, dev_err, grid, st)
                    : launch<FwdLseEpi<false, false>>(a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dlogits(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                           const DlogitsArgs& ea, bool has_bias, int* dev_err, int grid,
                           cudaStream_t st) {
  return has_bias ? launch<DlogitsEpi<true>>(a, b, g, ea, dev_err, grid, st)
                  : launch<DlogitsEpi<false>>(a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dw(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DwArgs& ea, int* dev_err, int grid, cudaStream_t st) {
  return launch<DwEpi>(a, b, g, ea, dev_err, grid, st);
}

cudaError_t launch_dx(const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DxArgs& ea, int* dev_err, int grid, cudaStream_t st) {
  return launch<DxEpi>(a, b, g, ea, dev_err, grid, st);
}

}  // namespace flce
