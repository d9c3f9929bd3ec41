// Internal interface between the C-ABI layer (flce_api.cu) and the kernel
// translation units (flce_gemm.cu, flce_rowwise.cu).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "gemm_engine.cuh"

namespace flce {

struct FwdLseArgs;
struct DlogitsArgs;
struct DwArgs;
struct DxArgs;

// GEMM kernel forms (flce_gemm.cu): one CTA per 128 x 256 tile, a CTA pair per
// 256 x 256 tile, or a CTA pair per 256 x 512 tile (the dx GEMM runs the wide
// form as 256 x 256 pairs). The pair forms need 128-row boxes in a K-major B
// map. `grid` is the CTA count of the single-CTA kernel (the SM count when it
// is the smaller).
// kGemmAuto is resolved per GEMM on the host before any launch.
enum GemmKind : int { kGemmSingle = 0, kGemmPair = 1, kGemmWide = 2, kGemmAuto = 3 };
// keep: the kept-block forward (FwdLseArgs.keep_*).
cudaError_t launch_fwd_lse(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const FwdLseArgs& ea, bool has_bias,
                           bool has_smooth, bool keep, int* dev_err, int grid, cudaStream_t st);
cudaError_t launch_dlogits(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmGeom& g, const DlogitsArgs& ea, bool has_bias, int* dev_err,
                           int grid, cudaStream_t st);
cudaError_t launch_dw(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
                      const DwArgs& ea, int* dev_err, int grid, cudaStream_t st);
cudaError_t launch_dx(GemmKind kind, const CUtensorMap& a, const CUtensorMap& b, const GemmGeom& g,
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
constexpr int kMergeRows = 32;   // token rows per merge block (one per lane)
constexpr int kMergeSplit = 8;   // warps per merge block, each folding every 8th vocab tile
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
  int fp16;          // operands are fp16: choose a power-of-two dL scale
  float* dl_scale;   // out [2]: factor applied to dL before rounding, and its inverse
  int* dev_err;
};
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st);

// Kept-probability backward (the kept block, and the stored mode, whose kept
// block spans the vocabulary): fp16 q [N, ld_q] relative to the running
// maxima of 32-column chunks chunk_max [ceil(Vb / 32), N] -> dL block
// [N, ld_dL] (bf16, or fp16 when fp16 = 1) and db partials
// [ceil(N / 32), ld_db]. q and dL may be the same buffer (converted in place).
struct ConvertArgs {
  const __half* q;
  int ld_q;
  const float* chunk_max;
  const float4* coef;
  const int64_t* y;
  int64_t y_off;
  int N, v0, Vb;
  uint16_t* dL;
  int ld_dL;
  int fp16;
  const float* dl_scale;
  float* db_part;  // null without a bias
  int ld_db;
};
cudaError_t launch_convert(const ConvertArgs& a, cudaStream_t st);
int convert_db_parts(int N);

// Vocabulary shards: local partials -> stats [4, N] = (m2, d, z_y or 0, sum z);
// rescale d by 2^(m2 - M) against the all-shard max M; fp32 -> bf16 cast.
struct ShardStatsArgs {
  const float* part_m;
  const float* part_d;
  const float* part_s;  // null without smoothing
  const float* zy;
  const int64_t* y;
  int N, NT;
  int64_t vocab_start, V, V_total, ignore_index;
  float* stats;
  int* dev_err;
};
cudaError_t launch_shard_stats(const ShardStatsArgs& a, cudaStream_t st);
cudaError_t launch_shard_rescale(float* stats, const float* gmax, int N, cudaStream_t st);
cudaError_t launch_cast16(const float* src, uint16_t* dst, int64_t n, bool fp16, cudaStream_t st);

cudaError_t launch_wait_timeout_selftest(int* dev_err, long long limit, cudaStream_t st);

cudaError_t launch_db_finalize(const float* db_part, int parts, int ld, int v0, int Vb, void* db,
                               bool db_fp32, bool fp16, cudaStream_t st);

}  // namespace flce
