// Epilogues of the FLCE GEMMs. Each call drains one 128 x 256 fp32 sub-tile
// of a CTA's TMEM accumulator, or the chunks of it that an EpiSlice names,
// with 128 threads (4 warps, one per TMEM lane quarter); thread i owns row i
// and reads it 32 columns at a time. tm and tn index the sub-tile in 128-row
// and 256-column units whatever the kernel's tile (a wide 256 x 512 tile is
// two sub-tiles per CTA on 8 warps, or on 16 with each sub-tile's columns
// split between two warps).
//
// Each epilogue states kWideWarps, the epilogue warps it runs with in the
// 256 x 512 kernel, and kStageNeed, the shared staging bytes a warp uses.
//
// Notation (fla fused_linear_cross_entropy.py; Liger-Kernel PR #239):
//   z = s * (acc + b_v)          logits of one token row, vocab column v
//   lse = log sum_v exp(z_v)      kept per (row, vocab tile) as base-2 (m, d)
//   dL = s * g * ((1 + 2 lam lse) p - eps/V - (1 - eps) [v == y]),  p = exp(z - lse)
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gemm_engine.cuh"

namespace flce {

constexpr float kLog2e = 1.4426950408889634f;

// Bias (bf16 or fp16 bits) of 32 consecutive vocab columns starting at
// col0 (< V); zero past V.
template <bool HAS_BIAS>
__device__ __forceinline__ void load_bias32(const uint16_t* __restrict__ bias, int col0, int V,
                                            float (&bv)[32], bool fp16) {
  if constexpr (!HAS_BIAS) {
#pragma unroll
    for (int j = 0; j < 32; ++j) bv[j] = 0.f;
  } else {
    if (col0 + 32 <= V) {
      const uint4* p = reinterpret_cast<const uint4*>(bias + col0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 u = __ldg(p + q);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          bv[q * 8 + 2 * e] = unpack_16(w[e] & 0xFFFFu, fp16);
          bv[q * 8 + 2 * e + 1] = unpack_16(w[e] >> 16, fp16);
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        bv[j] = (col0 + j < V) ? unpack_16(__ldg(bias + col0 + j), fp16) : 0.f;
    }
  }
}

// 32 fp32 values -> 64 bytes of the 16-bit operand type at dst (16-B aligned).
__device__ __forceinline__ void store32_16(void* dst, const float (&v)[32], bool fp16) {
  uint4* o = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_16x2(v[q * 8 + 0], v[q * 8 + 1], fp16);
    u.y = pack_16x2(v[q * 8 + 2], v[q * 8 + 3], fp16);
    u.z = pack_16x2(v[q * 8 + 4], v[q * 8 + 5], fp16);
    u.w = pack_16x2(v[q * 8 + 6], v[q * 8 + 7], fp16);
    o[q] = u;
  }
}

__device__ __forceinline__ uint16_t to16(float f, bool fp16) {
  return static_cast<uint16_t>(pack_16x2(f, 0.f, fp16) & 0xFFFFu);
}

// Column sums of a 32 x 32 block held one row per lane: afterwards lane L
// holds the sum over the warp of column L (recursive halving, 31 shuffles).
__device__ __forceinline__ float warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? v[i] : v[i + off];
      const float keep = upper ? v[i + off] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
  return v[0];
}

// Reductions of 32 values as trees (depth 4-5 instead of a 31-long dependent
// chain: with two epilogue warps per SM sub-partition the chain's latency is
// not hidden). The maximum and minimum take three inputs per instruction (16
// instructions; exact in any order). The sum adds packed pairs in the same
// association as the scalar tree t[i] = v[i] + v[i + 16], t[i] += t[i + w]
// for w = 8, 4, 2, 1 (16 instructions instead of 31, the same bits).
__device__ __forceinline__ float tree_max32(const float (&v)[32]) {
  float t[12];
#pragma unroll
  for (int k = 0; k < 10; ++k) t[k] = fmax3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  t[10] = v[30];
  t[11] = v[31];
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = fmax3(t[3 * k], t[3 * k + 1], t[3 * k + 2]);
  return fmaxf(fmax3(t[0], t[1], t[2]), t[3]);
}
__device__ __forceinline__ float tree_min32(const float (&v)[32]) {
  float t[12];
#pragma unroll
  for (int k = 0; k < 10; ++k) t[k] = fmin3(v[3 * k], v[3 * k + 1], v[3 * k + 2]);
  t[10] = v[30];
  t[11] = v[31];
#pragma unroll
  for (int k = 0; k < 4; ++k) t[k] = fmin3(t[3 * k], t[3 * k + 1], t[3 * k + 2]);
  return fminf(fmin3(t[0], t[1], t[2]), t[3]);
}
__device__ __forceinline__ float tree_sum32(const float (&v)[32]) {
  uint64_t t[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    t[i] = fadd2(f32x2(v[2 * i], v[2 * i + 1]), f32x2(v[2 * i + 16], v[2 * i + 17]));
#pragma unroll
  for (int w = 4; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fadd2(t[i], t[i + w]);
  float lo, hi;
  f32x2_split(t[0], lo, hi);
  return lo + hi;
}

// p ? a : b as one selp. A chain of selects that picks v[j] for j == k would
// otherwise be turned into the indexed load v[k], which puts v in local memory.
__device__ __forceinline__ float select_f32(bool p, float a, float b) {
  float r;
  asm("{\n\t.reg .pred q;\n\tsetp.ne.s32 q, %3, 0;\n\tselp.f32 %0, %1, %2, q;\n\t}"
      : "=f"(r)
      : "f"(a), "f"(b), "r"(static_cast<int>(p)));
  return r;
}

// ------------------------------------------------- asynchronous block stores
// A warp holds a 32 x 32 block one row per lane (v[j] = element (lane, j)).
// It writes the block into its own staging buffer in shared memory in the
// layout of a TMA box with the tensor map's swizzle (16-byte slots XOR-ed by
// row, which also keeps the writes free of bank conflicts), and one lane hands
// the box to the TMA engine. The global write then completes in the
// background, overlapping whatever the SM does next (in the 256 x 512 kernel,
// the next tile's MMAs); the tensor map clips rows and columns outside the
// output. The buffer is rewritten only once the previous store has read it;
// the kernel waits for all stores before it exits. (x, y) = (column, row) of
// the block's first element.
//   fp32   : 32 rows x 128 B, map swizzle 128B: slot q of row r at r*8 + (q ^ (r & 7))
//   16-bit : 32 rows x 64 B,  map swizzle 64B:  slot q of row r at r*4 + (q ^ ((r >> 1) & 3))
__device__ __forceinline__ void tma_block_f32(const CUtensorMap* map, int x, int y,
                                              const float (&v)[32], void* stage_raw, int lane) {
  float4* stage = static_cast<float4*>(stage_raw);
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 8; ++q)
    stage[lane * 8 + (q ^ (lane & 7))] =
        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stage, x, y);
    bulk_commit_group();
  }
}

__device__ __forceinline__ void tma_block_16(const CUtensorMap* map, int x, int y,
                                             const float (&v)[32], bool fp16, void* stage_raw,
                                             int lane) {
  uint4* stage = static_cast<uint4*>(stage_raw);
  if (lane == 0) bulk_wait_group_read0();
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 u;
    u.x = pack_16x2(v[8 * q + 0], v[8 * q + 1], fp16);
    u.y = pack_16x2(v[8 * q + 2], v[8 * q + 3], fp16);
    u.z = pack_16x2(v[8 * q + 4], v[8 * q + 5], fp16);
    u.w = pack_16x2(v[8 * q + 6], v[8 * q + 7], fp16);
    stage[lane * 4 + (q ^ ((lane >> 1) & 3))] = u;
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stage, x, y);
    bulk_commit_group();
  }
}

// ------------------------------------------------------------------ forward
// Folds each logits tile into per-(row, vocab tile) base-2 online-softmax
// partials (m = max z log2e, d = sum 2^(z log2e - m)), the tile's sum of z
// (label smoothing only) and the target logit z_y when y falls in the tile.
//
// KEEP (the kept-block forward): every 32-column chunk of the vocabulary
// columns [0, keep_cols) also leaves its probabilities relative to the running
// maximum after that chunk, q = 2^(z log2e - m_c) in (0, 1], as fp16 in the
// kept buffer (a TMA-stored [Ntok, keep_cols] view; these are the exponentials
// the online softmax computes anyway), and m_c in keep_max[chunk, row]. The
// backward turns them into that block's dL in place:
// p = q 2^(m_c - lse log2e).
struct FwdLseArgs {
  const uint16_t* bias;  // bf16 or fp16 bits
  int fp16;
  const int64_t* y;
  int64_t y_off;  // vocabulary id of W's first row (vocabulary shards; else 0)
  float scale;
  int V;
  int Ntok;
  float* part_m;  // [tiles_v, Ntok]
  float* part_d;  // [tiles_v, Ntok]
  float* part_s;  // [tiles_v, Ntok] or null
  float* zy;      // [Ntok]
  int keep_cols;         // KEEP: vocabulary columns kept (<= V)
  float* keep_max;       // KEEP: [ceil(keep_cols / 32), Ntok]
  CUtensorMap keep_map;  // KEEP: store map of the kept q, [Ntok, keep_cols] 16-bit
};

template <bool HAS_BIAS, bool HAS_SMOOTH, bool KEEP = false>
struct FwdLseEpi {
  static constexpr bool kAMN = false, kBMN = false;
  // With a bias and without smoothing, the kept variant spills at 16 warps.
  static constexpr int kWideWarps = (KEEP && HAS_BIAS && !HAS_SMOOTH) ? 8 : 16;
  static constexpr int kStageNeed = KEEP ? 32 * 32 * 2 : 0;  // one 16-bit 32 x 32 box
  using Args = FwdLseArgs;
  __device__ static void tile(const Args& a, const GemmGeom&, int tm, int tn, int row_in_tile,
                              int lane, int quad, uint32_t taddr, void* stage,
                              const EpiSlice& sl) {
    const int row = tm * kBM + row_in_tile;
    const int v0 = tn * kBN;
    const int64_t yv = row < a.Ntok ? __ldg(a.y + row) - a.y_off : -1;
    const int ty = (yv >= v0 && yv < static_cast<int64_t>(v0) + kBN) ? static_cast<int>(yv - v0) : -1;
    // With u = acc + b, z log2e = c2 u: one FFMA per logit feeds the ex2, and
    // a chunk's maximum of z log2e is c2 times its maximum of u (its minimum
    // when c2 < 0). S and the target logit are kept in units of u and scaled
    // once at the end.
    const float c2 = a.scale * kLog2e;
    const bool neg = c2 < 0.f;
    // The second warp of a column-split pair reuses its staging buffer (the
    // hand-off slots, and with KEEP the q boxes) only after its partner has
    // read the previous hand-off.
    if (sl.sub == 1 && sl.xcount > 0 &&
        !mbar_wait(sl.xfree, static_cast<uint32_t>((sl.xcount - 1) & 1), sl.abort_flag,
                   sl.dev_err))
      return;
    float m = -INFINITY, d = 0.f, S = 0.f, ut = 0.f;
#pragma unroll 1
    for (int c = sl.c_lo; c < sl.c_hi; ++c) {
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
      const int col0 = v0 + c * 32;
      const bool full = col0 + 32 <= a.V;  // the same for the whole warp
      if constexpr (HAS_BIAS) {
        float bv[32];
        load_bias32<true>(a.bias, col0 < a.V ? col0 : 0, a.V, bv, a.fp16 != 0);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += bv[j];
      }
      if ((ty >> 5) == c) {
#pragma unroll
        for (int j = 0; j < 32; ++j) ut = select_f32(j == (ty & 31), v[j], ut);
      }
      float cm;
      if (full) {
        if constexpr (HAS_SMOOTH) S += tree_sum32(v);
        cm = (neg ? tree_min32(v) : tree_max32(v)) * c2;
      } else {
        // The last vocabulary tile: columns >= V do not exist.
        cm = -INFINITY;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const bool ok = col0 + j < a.V;
          if constexpr (HAS_SMOOTH) S += ok ? v[j] : 0.f;
          cm = ok ? fmaxf(cm, v[j] * c2) : cm;
        }
      }
      const float nm = fmaxf(m, cm);
      if (nm != -INFINITY) {
        float acc = d * fast_exp2(m - nm);
        if (full) {
          // z log2e - nm for two logits per packed FFMA.
          const uint64_t c2x2 = f32x2(c2, c2), nmx2 = f32x2(-nm, -nm);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float lo, hi;
            f32x2_split(ffma2(f32x2(v[2 * j], v[2 * j + 1]), c2x2, nmx2), lo, hi);
            v[2 * j] = fast_exp2(lo);
            v[2 * j + 1] = fast_exp2(hi);
          }
          acc += tree_sum32(v);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float q = (col0 + j < a.V) ? fast_exp2(fmaf(v[j], c2, -nm)) : 0.f;
            if constexpr (KEEP) v[j] = q;
            acc += q;
          }
        }
        d = acc;
        m = nm;
      }
      if constexpr (KEEP) {
        // col0 < keep_cols <= V: the chunk has a real column, so nm is finite
        // and v holds its q. The map clips rows past Ntok and columns past
        // keep_cols. (The same for the whole warp.)
        if (col0 < a.keep_cols) {
          const int row0 = tm * kBM + quad * 32;
          if (row0 < a.Ntok) tma_block_16(&a.keep_map, col0, row0, v, true, stage, lane);
          if (row < a.Ntok) a.keep_max[static_cast<size_t>(col0 >> 5) * a.Ntok + row] = nm;
        }
      }
    }
    // The target column lies in at most one warp's chunks.
    const bool has_t = ty >= 0 && (ty >> 5) >= sl.c_lo && (ty >> 5) < sl.c_hi;
    if (row < a.Ntok && has_t) a.zy[row] = ut * a.scale;
    if (sl.sub == 1) {
      // Second half of a column-split sub-tile: hand (m, d, S) to the partner.
      // The hand-off slots are this warp's staging buffer: with KEEP, its last
      // q box must have been read out by the TMA engine first.
      if constexpr (KEEP) {
        if (lane == 0) bulk_wait_group_read0();
        __syncwarp();
      }
      sl.xchg[lane] = make_float4(m, d, S, 0.f);
      mbar_arrive(sl.xbar);
      return;
    }
    if (sl.sub == 0) {
      if (!mbar_wait(sl.xbar, sl.xph, sl.abort_flag, sl.dev_err)) return;
      const float4 o = sl.xchg[lane];
      mbar_arrive(sl.xfree);  // the partner may reuse its staging buffer
      const float nm = fmaxf(m, o.x);
      // A half whose columns all lie past V has m = -inf and d = 0.
      d = nm == -INFINITY ? 0.f : d * fast_exp2(m - nm) + o.y * fast_exp2(o.x - nm);
      m = nm;
      S += o.z;
    }
    if (row < a.Ntok) {
      const size_t o = static_cast<size_t>(tn) * a.Ntok + row;
      a.part_m[o] = m;
      a.part_d[o] = d;
      if constexpr (HAS_SMOOTH) a.part_s[o] = S * a.scale;
    }
  }
};

// ------------------------------------------------- backward: recompute + dL
// Recomputes a logits tile of the current vocab block, forms
// dL = a_n p - c_n - t_n [v == y_n] with per-row coefficients
// (lse2 = lse log2e, a = s g (1 + 2 lam lse), c = s g eps / V, t = s g (1 - eps)),
// writes it as bf16 into the staged block dL[Ntok, ld] and, with a bias,
// writes per-warp column sums (fp32, before rounding) for db.
struct DlogitsArgs {
  const uint16_t* bias;  // bf16 or fp16 bits
  int fp16;              // dL written as fp16 (else bf16), like the operands
  const float* dl_scale; // [0]: power-of-two factor applied to dL before rounding
  const int64_t* y;
  int64_t y_off;       // vocabulary id of W's first row (vocabulary shards; else 0)
  const float4* coef;  // [Ntok]: (lse2, a, c, t)
  float scale;
  int V;
  int Ntok;
  int v0;              // first vocab id of the block
  int Vb;              // vocab ids in the block
  float* db_part;      // [tiles_m * 4, ld_db] or null
  int ld_db;
  CUtensorMap dl_map;  // TMA store map of the dL block: [Ntok rows, Vb columns], 16-bit
};

template <bool HAS_BIAS>
struct DlogitsEpi {
  static constexpr bool kAMN = false, kBMN = false;
  // With a bias the db column sums need the registers of 8 warps (16 spill).
  static constexpr int kWideWarps = HAS_BIAS ? 8 : 16;
  static constexpr int kStageNeed = 32 * 32 * 2;  // one 16-bit 32 x 32 box
  using Args = DlogitsArgs;
  __device__ static void tile(const Args& a, const GemmGeom&, int tm, int tn, int row_in_tile,
                              int lane, int quad, uint32_t taddr, void* stage,
                              const EpiSlice& sl) {
    const int row = tm * kBM + row_in_tile;
    const int row0 = tm * kBM + quad * 32;  // the warp's first row (lane = row - row0)
    const bool row_ok = row < a.Ntok;
    const int vt0 = tn * kBN;  // block-relative
    const int vg0 = a.v0 + vt0;
    const float4 cf = row_ok ? __ldg(a.coef + row) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float dls = __ldg(a.dl_scale);
    const int64_t yv = row_ok ? __ldg(a.y + row) - a.y_off : -1;
    const int ty = (yv >= vg0 && yv < static_cast<int64_t>(vg0) + kBN) ? static_cast<int>(yv - vg0) : -1;
    // p = 2^(c2 (acc + b) - lse2) with c2 = s log2e: one FFMA per logit feeds
    // the ex2, one more gives a p - c; the target column subtracts t.
    const float c2 = a.scale * kLog2e;
#pragma unroll 1
    for (int c = sl.c_lo; c < sl.c_hi; ++c) {
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
      const int colb0 = vt0 + c * 32;
      const int colg0 = vg0 + c * 32;
      if constexpr (HAS_BIAS) {
        float bv[32];
        load_bias32<true>(a.bias, colg0 < a.V ? colg0 : 0, a.V, bv, a.fp16 != 0);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += bv[j];
      }
      {
        // a 2^(c2 u - lse2) - c for two logits per packed FFMA pair.
        const uint64_t c2x2 = f32x2(c2, c2), lx2 = f32x2(-cf.x, -cf.x);
        const uint64_t ax2 = f32x2(cf.y, cf.y), cx2 = f32x2(-cf.z, -cf.z);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float lo, hi;
          f32x2_split(ffma2(f32x2(v[2 * j], v[2 * j + 1]), c2x2, lx2), lo, hi);
          f32x2_split(ffma2(f32x2(fast_exp2(lo), fast_exp2(hi)), ax2, cx2), v[2 * j],
                      v[2 * j + 1]);
        }
      }
      if ((ty >> 5) == c) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] -= (j == (ty & 31)) ? cf.w : 0.f;
      }
      // Rows past N (their 2^(...) is not bounded) and columns past the block are 0.
      if (!row_ok) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = 0.f;
      }
      if (colb0 + 32 > a.Vb) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (colb0 + j < a.Vb) ? v[j] : 0.f;
      }
      if (row0 < a.Ntok && colb0 < a.Vb) {  // the same for the whole warp
        if (dls == 1.f) {
          tma_block_16(&a.dl_map, colb0, row0, v, a.fp16 != 0, stage, lane);
        } else {
          float sv[32];
          const uint64_t dx2 = f32x2(dls, dls);
#pragma unroll
          for (int j = 0; j < 16; ++j)
            f32x2_split(fmul2(f32x2(v[2 * j], v[2 * j + 1]), dx2), sv[2 * j], sv[2 * j + 1]);
          tma_block_16(&a.dl_map, colb0, row0, sv, a.fp16 != 0, stage, lane);
        }
      }
      if constexpr (HAS_BIAS) {
        const float colsum = warp_column_sums(v, lane);
        // A CTA pair's second half-tile can lie wholly past the last token
        // (odd count of 128-row tiles): it has no partial row of its own.
        if (colb0 + lane < a.Vb && tm * kBM < a.Ntok)
          a.db_part[static_cast<size_t>(tm * 4 + quad) * a.ld_db + colb0 + lane] = colsum;
      }
    }
  }
};

// ---------------------------------------------------------- backward: dW
// dW[v0 + r, :] = sum_n dL[n, r] x[n, :] for block-relative vocab row r.
struct DwArgs {
  CUtensorMap out_map;  // TMA store map of this block's dW rows: [Mrows, Ncols], fp32 or 16-bit
  int out_bf16;   // 1: dW is the 16-bit type (bf16, or fp16 when fp16)
  int fp16;
  const float* acc_scale;  // [0]: undoes the dL scale (power of two)
  int Mrows;      // Vb
  int Ncols;      // H
};

struct DwEpi {
  static constexpr bool kAMN = true, kBMN = true;
  static constexpr int kWideWarps = 8, kStageNeed = 32 * 32 * 4;  // one fp32 32 x 32 box
  using Args = DwArgs;
  __device__ static void tile(const Args& a, const GemmGeom&, int tm, int tn, int,
                              int lane, int quad, uint32_t taddr, void* stage,
                              const EpiSlice& sl) {
    const int r0 = tm * kBM + quad * 32;  // the warp's first block-relative row
    const float sc = __ldg(a.acc_scale);
#pragma unroll 1
    for (int c = sl.c_lo; c < sl.c_hi; ++c) {
      const int col0 = tn * kBN + c * 32;
      if (col0 >= a.Ncols) break;  // uniform over the warp
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
      if (sc != 1.f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= sc;
      }
      if (r0 >= a.Mrows) continue;  // the same for the whole warp
      if (a.out_bf16)
        tma_block_16(&a.out_map, col0, r0, v, a.fp16 != 0, stage, lane);
      else
        tma_block_f32(&a.out_map, col0, r0, v, stage, lane);
    }
  }
};

// ---------------------------------------------------------- backward: dx
// dx[n, :] accumulates sum over vocab blocks of dL_block[n, :] W_block in an
// fp32 buffer; the first block stores, the last one writes bf16 dx.
struct DxArgs {
  float* acc;             // [Ntok, ld] fp32 (unused when first && last)
  uint16_t* out;          // dx [Ntok, ld] bf16 / fp16 (fp32 when out_f32)
  int fp16;
  const float* acc_scale; // [0]: undoes the dL scale (power of two)
  int out_f32;            // last block writes fp32 (vocabulary-shard partial dx)
  int ld;                 // H
  int Ntok;
  int Ncols;              // H
  int first;
  int last;
};

struct DxEpi {
  static constexpr bool kAMN = false, kBMN = true;
  static constexpr int kWideWarps = 8, kStageNeed = 0;
  using Args = DxArgs;
  __device__ static void tile(const Args& a, const GemmGeom&, int tm, int tn, int row_in_tile,
                              int, int, uint32_t taddr, void*, const EpiSlice& sl) {
    const int row = tm * kBM + row_in_tile;
    const bool row_ok = row < a.Ntok;
    const size_t orow = static_cast<size_t>(row_ok ? row : 0) * a.ld;
    const float sc = __ldg(a.acc_scale);
#pragma unroll 1
    for (int c = sl.c_lo; c < sl.c_hi; ++c) {
      float v[32];
      tmem_ld_32cols(taddr + c * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] *= sc;
      const int col0 = tn * kBN + c * 32;
      if (row_ok && col0 < a.Ncols) accumulate(a, orow, col0, v);
    }
  }
  __device__ __forceinline__ static void accumulate(const Args& a, size_t orow, int col0,
                                                   float (&v)[32]) {
    {
      const int ncol = min(32, a.Ncols - col0);
      float* accp = a.acc + orow + col0;
      if (ncol == 32) {
        if (!a.first) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 p = reinterpret_cast<const float4*>(accp)[q];
            v[4 * q] += p.x;
            v[4 * q + 1] += p.y;
            v[4 * q + 2] += p.z;
            v[4 * q + 3] += p.w;
          }
        }
        if (a.last && a.out_f32) {
          float* o = reinterpret_cast<float*>(a.out) + orow + col0;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(o)[q] =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else if (a.last) {
          store32_16(a.out + orow + col0, v, a.fp16 != 0);
        } else {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            reinterpret_cast<float4*>(accp)[q] =
                make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < ncol) {
            const float val = v[j] + (a.first ? 0.f : accp[j]);
            if (a.last && a.out_f32)
              reinterpret_cast<float*>(a.out)[orow + col0 + j] = val;
            else if (a.last)
              a.out[orow + col0 + j] = to16(val, a.fp16 != 0);
            else
              accp[j] = val;
          }
        }
      }
    }
  }
};

}  // namespace flce
