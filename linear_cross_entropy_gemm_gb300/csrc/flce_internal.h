// Internal interface between the C-ABI layer (flce_api.cu) and the kernel
// translation units (flce_gemm.cu, flce_rowwise.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gemm_engine.cuh"

namespace flce {

struct FwdLseArgs;
struct DlogitsArgs;
struct DwArgs;
struct DxArgs;

// Persistent tcgen05 GEMMs (flce_gemm.cu). pair = CTA-pair kernel (256 x 256
// tiles; a K-major B map must then have 128-row boxes). `grid` is the CTA
// count of the single-CTA kernel (the SM count when it is the smaller).
cudaError_t launch_fwd_lse(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const FwdLseArgs& ea, bool has_bias,
                           bool has_smooth, int* dev_err, int grid, cudaStream_t st);
cudaError_t launch_dlogits(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const DlogitsArgs& ea, bool has_bias, int* dev_err,
                           int grid, cudaStream_t st);
cudaError_t launch_dw(bool pair, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DwArgs& ea, int* dev_err, int grid, cudaStream_t st);
cudaError_t launch_dx(bool pair, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DxArgs& ea, int* dev_err, int grid, cudaStream_t st);

// Row-wise kernels (flce_rowwise.cu).
struct MergeArgs {
  const float* part_m;
  const float* part_d;
  const float* part_s;  // null without label smoothing
  const float* zy;
  const int64_t* y;
  int N, NT, V;
  int64_t ignore_index;
  float eps, lam;
  int reduction;
  float* lse;
  float* loss;          // [N] (none) or [1]
  double* blk_sum;      // [blocks] (sum / mean)
  int* blk_cnt;         // [blocks]
  int* dev_err;
};
constexpr int kMergeThreads = 256;
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st);
cudaError_t launch_finalize(const MergeArgs& a, cudaStream_t st);

struct PrepArgs {
  const float* dloss;
  const float* lse;
  const int64_t* y;
  int N, V;
  int64_t ignore_index;
  float eps, lam, scale;
  int reduction;
  float4* coef;
  int* dev_err;
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st);

cudaError_t launch_db_finalize(const float* db_part, int parts, int ld, int v0, int Vb, void* db,
                               bool db_fp32, cudaStream_t st);

}  // namespace flce
