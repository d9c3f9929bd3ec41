// Row-wise (HBM-bound) kernels of the FLCE path:
//   merge     : fold the per-vocab-tile (m, d) partials of each token into
//               lse = m + log d, then the per-token loss and its reduction
//   finalize  : deterministic sum of the per-block loss partials
//   prep      : per-token backward coefficients (upstream gradient, z-loss,
//               smoothing) so the dlogits epilogue is a couple of FMAs
//   db        : ordered sum of the per-warp bias-gradient partials
#include <cuda_fp16.h>
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

// Folds one token row's per-vocab-tile base-2 partials (m_t, d_t, S_t) into
// M = max m_t, D = sum d_t 2^(m_t - M), S = sum S_t, in the one fixed order
// both the loss merge and the vocabulary-shard statistics use (so a single
// shard reproduces the plain call bit for bit). A block takes kMergeRows rows
// (lane = row: each load of one vocab tile's partials is one coalesced
// 128-byte segment); warp w folds tiles w, w + kMergeSplit, ...; warp 0 then
// merges the kMergeSplit results in warp order. Returns true in warp 0, whose
// M, D, S hold the row's result; the other warps may leave.
__device__ __forceinline__ bool fold_partials(const float* part_m, const float* part_d,
                                              const float* part_s, int N, int NT, float& M,
                                              float& D, float& S) {
  __shared__ float sm[kMergeSplit][kMergeRows], sd[kMergeSplit][kMergeRows],
      ss[kMergeSplit][kMergeRows];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int row = blockIdx.x * kMergeRows + lane;
  M = -INFINITY;
  D = 0.f;
  S = 0.f;
  if (row < N) {
#pragma unroll 4
    for (int t = w; t < NT; t += kMergeSplit) {
      const size_t o = static_cast<size_t>(t) * N + row;
      const float m = __ldg(part_m + o);
      const float d = __ldg(part_d + o);
      const float nm = fmaxf(M, m);
      D = D * fast_exp2(M - nm) + d * fast_exp2(m - nm);
      M = nm;
      if (part_s) S += __ldg(part_s + o);
    }
  }
  sm[w][lane] = M;
  sd[w][lane] = D;
  ss[w][lane] = S;
  __syncthreads();
  if (w != 0) return false;
  M = sm[0][lane];
  D = sd[0][lane];
  S = ss[0][lane];
#pragma unroll
  for (int k = 1; k < kMergeSplit; ++k) {
    const float m = sm[k][lane];
    const float nm = fmaxf(M, m);
    if (nm != -INFINITY) {  // a warp with no vocab tile keeps (-inf, 0)
      D = D * fast_exp2(M - nm) + sd[k][lane] * fast_exp2(m - nm);
      M = nm;
    }
    S += ss[k][lane];
  }
  return true;
}

// lse = (M + log2 D) ln 2 (the (m, d) merge of online softmax), then the
// per-token loss and, for sum / mean, the block's loss sum (fixed order).
template <bool HAS_SMOOTH>
__global__ void __launch_bounds__(kMergeRows * kMergeSplit) merge_kernel(const MergeArgs a) {
  float M, D, S;
  if (!fold_partials(a.part_m, a.part_d, HAS_SMOOTH ? a.part_s : nullptr, a.N, a.NT, M, D, S))
    return;
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kMergeRows + lane;
  double l = 0.0;
  int valid = 0;
  if (row < a.N) {
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
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      l += __shfl_down_sync(0xffffffffu, l, o);
      valid += __shfl_down_sync(0xffffffffu, valid, o);
    }
    if (lane == 0) {
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
  const int blocks = (a.N + kMergeRows - 1) / kMergeRows;
  if (a.part_s)
    merge_kernel<true><<<blocks, kMergeRows * kMergeSplit, 0, st>>>(a);
  else
    merge_kernel<false><<<blocks, kMergeRows * kMergeSplit, 0, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const MergeArgs& a, cudaStream_t st) {
  const int blocks = (a.N + kMergeRows - 1) / kMergeRows;
  finalize_loss_kernel<<<1, 1024, 0, st>>>(a.blk_sum, a.blk_cnt, blocks, a.reduction, a.loss);
  return cudaGetLastError();
}

// One block: count the non-ignored tokens, then per token
//   g    = dloss (sum) | dloss / total (mean) | dloss[n] (none); 0 if ignored
//   coef = (lse log2e, s g (1 + 2 lam lse), s g eps / V, s g (1 - eps)).
// With fp16 operands dL is stored scaled by 2^k so that its bound
// max_n (|a_n| + |c_n| + |t_n|) (p <= 1) sits near 2^14: large loss scales do
// not overflow fp16 and small gradients do not flush to zero. The backward
// GEMM epilogues multiply by 2^-k in fp32 (exact).
__global__ void __launch_bounds__(1024) prep_kernel(const PrepArgs a) {
  double unused = 0.0;
  int cnt = 0;
  for (int i = threadIdx.x; i < a.N; i += blockDim.x) cnt += (a.y[i] != a.ignore_index);
  block_sum(unused, cnt);
  float bound = 0.f;
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
    const float4 cf = make_float4(lse * kLog2eF, sg * (1.f + 2.f * a.lam * lse),
                                  sg * (a.eps / a.V), sg * (1.f - a.eps));
    a.coef[i] = cf;
    bound = fmaxf(bound, fabsf(cf.y) + fabsf(cf.z) + fabsf(cf.w));
  }
  // Block max of the bound (fixed order) -> the dL scale.
  __shared__ float smax[32];
  for (int o = 16; o > 0; o >>= 1) bound = fmaxf(bound, __shfl_xor_sync(0xffffffffu, bound, o));
  if ((threadIdx.x & 31) == 0) smax[threadIdx.x >> 5] = bound;
  __syncthreads();
  if (threadIdx.x == 0) {
    float mx = 0.f;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) mx = fmaxf(mx, smax[w]);
    int k = 0;
    if (a.fp16 && mx > 0.f && mx < INFINITY) {
      int e;
      frexpf(mx, &e);        // mx = f 2^e, f in [0.5, 1)
      k = 14 - e;            // bound * 2^k in [2^13, 2^14)
      k = max(-100, min(100, k));
    }
    a.dl_scale[0] = ldexpf(1.f, k);
    a.dl_scale[1] = ldexpf(1.f, -k);
  }
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st) {
  prep_kernel<<<1, 1024, 0, st>>>(a);
  return cudaGetLastError();
}

// db[v0 + c] = sum over the partial rows p of part[p, c]. A block takes 32
// columns (one coalesced 128-byte segment per partial row) and its 8 warps
// split the partial rows: warp w sums rows w, w + 8, ... in order, with eight
// independent loads in flight per thread; warp 0 then adds the 8 warp sums in
// warp order. A fixed order throughout: deterministic.
constexpr int kDbWarps = 8;
__global__ void __launch_bounds__(32 * kDbWarps) db_finalize_kernel(
    const float* __restrict__ part, int parts, int ld, int v0, int Vb, void* db, int db_fp32,
    int fp16) {
  __shared__ float s_sum[kDbWarps][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (c < Vb) {
    int p = w;
    for (; p + 7 * kDbWarps < parts; p += 8 * kDbWarps) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = __ldg(part + static_cast<size_t>(p + k * kDbWarps) * ld + c);
#pragma unroll
      for (int k = 0; k < 8; ++k) s += v[k];
    }
    for (; p < parts; p += kDbWarps) s += __ldg(part + static_cast<size_t>(p) * ld + c);
  }
  s_sum[w][lane] = s;
  __syncthreads();
  if (w != 0 || c >= Vb) return;
  float t = s_sum[0][lane];
#pragma unroll
  for (int k = 1; k < kDbWarps; ++k) t += s_sum[k][lane];
  if (db_fp32)
    reinterpret_cast<float*>(db)[v0 + c] = t;
  else
    reinterpret_cast<uint16_t*>(db)[v0 + c] =
        static_cast<uint16_t>(pack_16x2(t, 0.f, fp16 != 0) & 0xFFFFu);
}

cudaError_t launch_db_finalize(const float* db_part, int parts, int ld, int v0, int Vb, void* db,
                               bool db_fp32, bool fp16, cudaStream_t st) {
  db_finalize_kernel<<<(Vb + 31) / 32, 32 * kDbWarps, 0, st>>>(db_part, parts, ld, v0, Vb, db,
                                                              db_fp32 ? 1 : 0, fp16 ? 1 : 0);
  return cudaGetLastError();
}

// Kept-probability backward: dL[n, v] = a_n q[n, v] 2^(m_c(n, v) - lse2_n)
//   - c_n - t_n [v == y_n] for the vocab block [v0, v0 + Vb), q being the
// forward's fp16 2^(z log2e - m_c) and m_c the running maximum of the row's
// logits after the 32-column chunk that holds v (flce_forward_keep). One CTA
// covers 32 tokens x one 256-column vocab tile. Thread i owns 8 columns
// (16-byte loads and stores; one chunk) of rows i/32, i/32 + 4, ..., so
// eight independent loads are in flight per thread; the fp32 column sums over
// the 32 tokens (db partials, row blockIdx.y) are combined through shared
// memory. The conversion runs in place (q and dL are the same buffer), so q is
// read with plain loads: each thread reads its 16 bytes before it overwrites
// them and no other thread touches them.
constexpr int kConvRows = 32;
constexpr int kConvRowGroups = 4;  // 128 threads = 32 column groups x 4 row groups
__global__ void __launch_bounds__(128) probs_to_dlogits_kernel(const ConvertArgs a) {
  // Per (chunk, row): the factor a 2^(m_c - lse2).
  __shared__ float s_scale[8][kConvRows];
  __shared__ float s_c[kConvRows], s_t[kConvRows];
  __shared__ int s_ty[kConvRows];
  __shared__ float s_sum[kConvRowGroups][256];
  const int tile = blockIdx.x;  // 256-column tile inside the block
  const int r0 = blockIdx.y * kConvRows;
  const int cg = threadIdx.x & 31;
  const int rg = threadIdx.x >> 5;
  const int colb = tile * 256 + cg * 8;  // block-relative first column of this thread
  if (threadIdx.x < kConvRows) {
    const int r = r0 + threadIdx.x;
    float c = 0.f, t = 0.f;
    int ty = -1;
    if (r < a.N) {
      const float4 cf = a.coef[r];
      c = cf.z;
      t = cf.w;
      const int64_t yv = a.y[r] - a.y_off;
      const int64_t lo = static_cast<int64_t>(a.v0) + tile * 256;
      if (yv >= lo && yv < lo + 256) ty = static_cast<int>(yv - a.v0);
    }
    s_c[threadIdx.x] = c;
    s_t[threadIdx.x] = t;
    s_ty[threadIdx.x] = ty;
  }
  {
    // 8 chunks x 32 rows of maxima, two per thread (each chunk's 32 rows are
    // one coalesced 128-byte load).
    const int nchunks = (a.Vb + 31) / 32;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int i = threadIdx.x + 128 * k;
      const int ch = i >> 5, rr = i & 31;
      const int r = r0 + rr, cidx = tile * 8 + ch;
      float sc = 0.f;
      if (r < a.N && cidx < nchunks) {
        const float4 cf = a.coef[r];
        sc = cf.y * exp2f(a.chunk_max[static_cast<size_t>(cidx) * a.N + r] - cf.x);
      }
      s_scale[ch][rr] = sc;
    }
  }
  __syncthreads();
  const float dls = a.dl_scale[0];
  const bool f16 = a.fp16 != 0;
  float sum[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) sum[j] = 0.f;
  uint4 q[kConvRows / kConvRowGroups];
#pragma unroll
  for (int k = 0; k < kConvRows / kConvRowGroups; ++k) {
    const int i = rg + kConvRowGroups * k;
    if (r0 + i < a.N && colb < a.Vb)
      q[k] = *reinterpret_cast<const uint4*>(a.q + static_cast<size_t>(r0 + i) * a.ld_q + a.v0 +
                                             colb);
  }
#pragma unroll
  for (int k = 0; k < kConvRows / kConvRowGroups; ++k) {
    const int i = rg + kConvRowGroups * k;
    if (r0 + i >= a.N || colb >= a.Vb) continue;
    const uint32_t w[4] = {q[k].x, q[k].y, q[k].z, q[k].w};
    const float scale = s_scale[cg >> 2][i];
    float d[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
      d[2 * e] = f.x;
      d[2 * e + 1] = f.y;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float v = fmaf(scale, d[j], -s_c[i]) - (colb + j == s_ty[i] ? s_t[i] : 0.f);
      v = colb + j < a.Vb ? v : 0.f;
      sum[j] += v;
      d[j] = v * dls;
    }
    uint4 o;
    o.x = pack_16x2(d[0], d[1], f16);
    o.y = pack_16x2(d[2], d[3], f16);
    o.z = pack_16x2(d[4], d[5], f16);
    o.w = pack_16x2(d[6], d[7], f16);
    *reinterpret_cast<uint4*>(a.dL + static_cast<size_t>(r0 + i) * a.ld_dL + colb) = o;
  }
  if (a.db_part) {
#pragma unroll
    for (int j = 0; j < 8; ++j) s_sum[rg][cg * 8 + j] = sum[j];
    __syncthreads();
    // Fixed order over the four row groups: deterministic.
    for (int c = threadIdx.x; c < 256; c += blockDim.x) {
      const float tot = ((s_sum[0][c] + s_sum[1][c]) + s_sum[2][c]) + s_sum[3][c];
      if (tile * 256 + c < a.Vb)
        a.db_part[static_cast<size_t>(blockIdx.y) * a.ld_db + tile * 256 + c] = tot;
    }
  }
}

cudaError_t launch_convert(const ConvertArgs& a, cudaStream_t st) {
  dim3 grid((a.Vb + 255) / 256, (a.N + kConvRows - 1) / kConvRows);
  probs_to_dlogits_kernel<<<grid, 128, 0, st>>>(a);
  return cudaGetLastError();
}

int convert_db_parts(int N) { return (N + kConvRows - 1) / kConvRows; }

// One shard's per-token statistics over its vocabulary rows: the (m, d)
// merge of its tile partials, its sum of z, and z_y when the target falls in
// the shard (0 otherwise, so a SUM across shards yields z_y exactly once).
__global__ void __launch_bounds__(kMergeRows * kMergeSplit)
    shard_stats_kernel(const ShardStatsArgs a) {
  float M, D, S;
  if (!fold_partials(a.part_m, a.part_d, a.part_s, a.N, a.NT, M, D, S)) return;
  const int row = blockIdx.x * kMergeRows + (threadIdx.x & 31);
  if (row >= a.N) return;
  const int64_t yv = a.y[row];
  float zy = 0.f;
  if (yv != a.ignore_index) {
    if (yv < 0 || yv >= a.V_total) {
      if (a.dev_err) atomicOr(a.dev_err, kDevErrTarget);
    } else if (yv >= a.vocab_start && yv < a.vocab_start + a.V) {
      zy = a.zy[row];
    }
  }
  a.stats[row] = M;
  a.stats[static_cast<size_t>(a.N) + row] = D;
  a.stats[2 * static_cast<size_t>(a.N) + row] = zy;
  a.stats[3 * static_cast<size_t>(a.N) + row] = S;
}

cudaError_t launch_shard_stats(const ShardStatsArgs& a, cudaStream_t st) {
  shard_stats_kernel<<<(a.N + kMergeRows - 1) / kMergeRows, kMergeRows * kMergeSplit, 0, st>>>(a);
  return cudaGetLastError();
}

// d <- d 2^(m - M), m <- M, with M the maximum of m over all shards.
__global__ void shard_rescale_kernel(float* stats, const float* gmax, int N) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= N) return;
  const float M = gmax[row];
  const float m = stats[row];
  stats[static_cast<size_t>(N) + row] *= fast_exp2(m - M);
  stats[row] = M;
}

cudaError_t launch_shard_rescale(float* stats, const float* gmax, int N, cudaStream_t st) {
  shard_rescale_kernel<<<(N + 255) / 256, 256, 0, st>>>(stats, gmax, N);
  return cudaGetLastError();
}

__global__ void cast16_kernel(const float* __restrict__ src, uint16_t* __restrict__ dst, int64_t n,
                              int fp16) {
  const int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4;
  if (i + 4 <= n) {
    const float4 v = *reinterpret_cast<const float4*>(src + i);
    uint2 o;
    o.x = pack_16x2(v.x, v.y, fp16 != 0);
    o.y = pack_16x2(v.z, v.w, fp16 != 0);
    *reinterpret_cast<uint2*>(dst + i) = o;
  } else {
    for (int64_t j = i; j < n; ++j)
      dst[j] = static_cast<uint16_t>(pack_16x2(src[j], 0.f, fp16 != 0) & 0xFFFFu);
  }
}

cudaError_t launch_cast16(const float* src, uint16_t* dst, int64_t n, bool fp16, cudaStream_t st) {
  const int64_t blocks = (n + 1023) / 1024;
  if (blocks == 0) return cudaSuccess;
  cast16_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(src, dst, n, fp16 ? 1 : 0);
  return cudaGetLastError();
}

// Failure-detection self-test: one thread waits, through the same bounded
// mbar_wait the GEMM pipelines use, on an mbarrier that nothing arrives on.
// The wait gives up after `limit` cycles and sets the timeout bit in dev_err;
// the kernel then returns normally and the context stays usable.
__global__ void wait_timeout_selftest_kernel(int* dev_err, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, dev_err, limit);
}

cudaError_t launch_wait_timeout_selftest(int* dev_err, long long limit, cudaStream_t st) {
  wait_timeout_selftest_kernel<<<1, 32, 0, st>>>(dev_err, limit);
  return cudaGetLastError();
}

}  // namespace flce
