// Row-wise (HBM-bound) kernels of the FLCE path:
//   merge     : fold the per-vocab-tile (m, d) partials of each token into
//               lse = m + log d, then the per-token loss and its reduction
//   finalize  : deterministic sum of the per-block loss partials
//   prep      : per-token backward coefficients (upstream gradient, z-loss,
//               smoothing) so the dlogits epilogue is a couple of FMAs
//   db        : ordered sum of the per-warp bias-gradient partials
#include <cuda_runtime.h>

#include "flce_internal.h"
#include "sm103_primitives.cuh"

namespace flce {

constexpr double kLn2 = 0.69314718055994530942;
constexpr float kLog2eF = 1.4426950408889634f;

// Block-wide sum of a double and an int over blockDim.x (a multiple of 32)
// threads in a fixed order. Result valid in thread 0.
__device__ __forceinline__ void block_sum(double& v, int& c) {
  __shared__ double sv[32];
  __shared__ int sc[32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v += __shfl_down_sync(0xffffffffu, v, o);
    c += __shfl_down_sync(0xffffffffu, c, o);
  }
  if (lane == 0) {
    sv[w] = v;
    sc[w] = c;
  }
  __syncthreads();
  if (w == 0) {
    const int nw = blockDim.x >> 5;
    v = lane < nw ? sv[lane] : 0.0;
    c = lane < nw ? sc[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      v += __shfl_down_sync(0xffffffffu, v, o);
      c += __shfl_down_sync(0xffffffffu, c, o);
    }
  }
  __syncthreads();
}

// lse from base-2 partials: M = max m_t, D = sum d_t 2^(m_t - M),
// lse = (M + log2 D) ln 2 (the (m, d) merge of online softmax).
template <bool HAS_SMOOTH>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const MergeArgs a) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  double l = 0.0;
  int valid = 0;
  if (row < a.N) {
    float M = -INFINITY, D = 0.f, S = 0.f;
    const float* pm = a.part_m + row;
    const float* pd = a.part_d + row;
    for (int t = 0; t < a.NT; ++t) {
      const size_t o = static_cast<size_t>(t) * a.N;
      const float m = __ldg(pm + o);
      const float d = __ldg(pd + o);
      const float nm = fmaxf(M, m);
      D = D * fast_exp2(M - nm) + d * fast_exp2(m - nm);
      M = nm;
      if constexpr (HAS_SMOOTH) S += __ldg(a.part_s + row + o);
    }
    const double lse = (static_cast<double>(M) + log2(static_cast<double>(D))) * kLn2;
    a.lse[row] = static_cast<float>(lse);
    const int64_t yv = a.y[row];
    if (yv != a.ignore_index) {
      valid = 1;
      if (yv < 0 || yv >= a.V) {
        if (a.dev_err) atomicOr(a.dev_err, kDevErrTarget);
      } else {
        const double eps = a.eps;
        l = (1.0 - eps) * (lse - static_cast<double>(a.zy[row])) + eps * lse +
            static_cast<double>(a.lam) * lse * lse;
        if constexpr (HAS_SMOOTH) l -= eps / a.V * static_cast<double>(S);
      }
    }
    if (a.reduction == 0) a.loss[row] = static_cast<float>(l);
  }
  if (a.reduction != 0) {
    block_sum(l, valid);
    if (threadIdx.x == 0) {
      a.blk_sum[blockIdx.x] = l;
      a.blk_cnt[blockIdx.x] = valid;
    }
  }
}

__global__ void finalize_loss_kernel(const double* blk_sum, const int* blk_cnt, int nblk,
                                     int reduction, float* loss) {
  double v = 0.0;
  int c = 0;
  for (int i = threadIdx.x; i < nblk; i += blockDim.x) {
    v += blk_sum[i];
    c += blk_cnt[i];
  }
  block_sum(v, c);
  if (threadIdx.x == 0) {
    if (reduction == 2) v = c > 0 ? v / c : 0.0;
    loss[0] = static_cast<float>(v);
  }
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t st) {
  const int blocks = (a.N + kMergeThreads - 1) / kMergeThreads;
  if (a.part_s)
    merge_kernel<true><<<blocks, kMergeThreads, 0, st>>>(a);
  else
    merge_kernel<false><<<blocks, kMergeThreads, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const MergeArgs& a, cudaStream_t st) {
  const int blocks = (a.N + kMergeThreads - 1) / kMergeThreads;
  finalize_loss_kernel<<<1, 1024, 0, st>>>(a.blk_sum, a.blk_cnt, blocks, a.reduction, a.loss);
  return cudaGetLastError();
}

// One block: count the non-ignored tokens, then per token
//   g    = dloss (sum) | dloss / total (mean) | dloss[n] (none); 0 if ignored
//   coef = (lse log2e, s g (1 + 2 lam lse), s g eps / V, s g (1 - eps)).
__global__ void __launch_bounds__(1024) prep_kernel(const PrepArgs a) {
  double unused = 0.0;
  int cnt = 0;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) cnt += (a.y[i] != a.ignore_index);
  block_sum(unused, cnt);
  __shared__ float g_all;
  if (threadIdx.x == 0) {
    const float d0 = a.dloss[0];
    g_all = (a.reduction == 2) ? (cnt > 0 ? static_cast<float>(static_cast<double>(d0) / cnt) : 0.f)
                               : d0;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) {
    const int64_t yv = a.y[i];
    float g = (a.reduction == 0) ? a.dloss[i] : g_all;
    if (yv == a.ignore_index) {
      g = 0.f;
    } else if (yv < 0 || yv >= a.V) {
      if (a.dev_err) atomicOr(a.dev_err, kDevErrTarget);
      g = 0.f;
    }
    const float lse = a.lse[i];
    const float sg = a.scale * g;
    a.coef[i] = make_float4(lse * kLog2eF, sg * (1.f + 2.f * a.lam * lse), sg * (a.eps / a.V),
                            sg * (1.f - a.eps));
  }
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st) {
  prep_kernel<<<1, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

__global__ void db_finalize_kernel(const float* __restrict__ part, int parts, int ld, int v0,
                                   int Vb, void* db, int db_fp32) {
  const int c = blockIdx.x * blockDim.x + threadIdx.x;
  if (c >= Vb) return;
  float s = 0.f;
  for (int p = 0; p < parts; ++p) s += part[static_cast<size_t>(p) * ld + c];
  if (db_fp32)
    reinterpret_cast<float*>(db)[v0 + c] = s;
  else
    reinterpret_cast<__nv_bfloat16*>(db)[v0 + c] = __float2bfloat16_rn(s);
}

cudaError_t launch_db_finalize(const float* db_part, int parts, int ld, int v0, int Vb, void* db,
                               bool db_fp32, cudaStream_t st) {
  db_finalize_kernel<<<(Vb + 255) / 256, 256, 0, st>>>(db_part, parts, ld, v0, Vb, db,
                                                       db_fp32 ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace flce
