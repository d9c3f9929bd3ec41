// C ABI of the FLCE library (declared in include/flce.h): argument checks,
// workspace carving, TMA descriptor encoding and the launch sequence.
//
// Forward  (DeepSpeed PR #8792 "What": forward keeps per-token softmax
//           statistics only):
//   fwd_lse GEMM  x W^T tile by tile -> (m, d[, sum z]) partials + z_y; in the
//                 kept-block mode also the kept block's fp16 probabilities
//                 (the first backward block, or keep_vocab columns) and their
//                 32-column running maxima
//   merge         partials -> lse, per-token loss, reduction
// Backward (same page: logits recomputed one vocabulary block at a time, so
//           each dW block is one GEMM over all tokens):
//   prep          per-token coefficients from dloss, lse, y
//   per vocab block [v0, v0 + Vb):
//     dlogits GEMM  recompute x W_blk^T -> dL_blk = s dz (bf16) + db partials,
//                   or, for the kept block, the in-place conversion of its
//                   kept probabilities
//     dW GEMM       dW[v0:v0+Vb] = dL_blk^T x            (K = all tokens)
//     dx GEMM       dx (+)= dL_blk W_blk                  (fp32 across blocks)
//     db finalize   (with a bias)
// The stored-probability mode is the kept-block mode with one block over the
// whole vocabulary; keep_vocab sets any width in between.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include "../../include/flce.h"
#include "epilogues.cuh"
#include "flce_internal.h"

using namespace flce;

namespace {

// Default backward vocabulary block: the widest multiple of 256 whose staged
// dL block [N, BVc] fits kDlBudgetBytes (fewer, larger dW / dx GEMMs: less
// wave-quantisation tail and fewer fp32 dx read-modify-writes), at least
// kMinVocabBlock.
constexpr int64_t kDlBudgetBytes = 1LL << 30;
constexpr int64_t kMinVocabBlock = 4096;
constexpr size_t kAlign = 256;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// 2-D 16-bit tensor [outer, inner] (bf16, or fp16 when fp16) with row pitch
// `pitch_bytes`, 128-B swizzled boxes of box_inner x box_outer elements;
// out-of-range elements read as 0.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
               uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer, bool fp16) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA store map of a row-major [outer, inner] output for the epilogues'
// 32 x 32 blocks: fp32 with the 128-byte swizzle (128-byte box rows) or a
// 16-bit type with the 64-byte swizzle (64-byte box rows), the staging layouts
// of epilogues.cuh. Stores are clipped to [inner, outer].
bool encode_store_2d(CUtensorMap* m, void* base, uint64_t inner, uint64_t outer,
                     uint64_t pitch_bytes, bool fp32) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, fp32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base,
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            fp32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int cdiv(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// GEMM kernel form of a call: an explicit gemm_form decides; with the
// default form, FLCE_GEMM_FORM=single|pair|wide in the environment overrides
// the library default (for A/B measurements), which is chosen per GEMM
// (gemm_for). All forms compute identical results up to the order of fp32
// accumulation inside a tile.
GemmKind gemm_kind(const flce_params_t* p) {
  switch (p->gemm_form) {
    case FLCE_GEMM_SINGLE_CTA: return kGemmSingle;
    case FLCE_GEMM_CTA_PAIR: return kGemmPair;
    case FLCE_GEMM_WIDE_PAIR: return kGemmWide;
    default: break;
  }
  const char* e = std::getenv("FLCE_GEMM_FORM");
  if (e && std::strcmp(e, "single") == 0) return kGemmSingle;
  if (e && std::strcmp(e, "pair") == 0) return kGemmPair;
  if (e && std::strcmp(e, "wide") == 0) return kGemmWide;
  return kGemmAuto;
}

// The default form of one GEMM D[M, N] = A[M, K] B[N, K]^T. The wide tile's
// epilogue is not overlapped, so it pays only when the K loop is long enough
// to amortise it, and its tiles are twice as large, so it needs enough of them
// to fill the GPU's 76 clusters. Otherwise the 256 x 256 pair is used.
// Measured on GB300: at K = 4096 (Llama-3 head) the wide step is 2 % faster
// under the power cap; at K = 2048 the wide forward is 7-16 % slower.
constexpr int64_t kWideMinK = 4096;
constexpr int64_t kWideMinTiles = 8 * 76;
GemmKind gemm_for(GemmKind kind, int64_t M, int64_t N, int64_t K) {
  if (kind != kGemmAuto) return kind;
  const int64_t wide_tiles = ((M + 255) / 256) * ((N + 511) / 512);
  return (K >= kWideMinK && wide_tiles >= kWideMinTiles) ? kGemmWide : kGemmPair;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// SM count and architecture of the current device.
flce_status_t device_info(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (major != 10 || minor != 3) return FLCE_ERR_UNSUPPORTED;
  return FLCE_OK;
}

flce_status_t check_params(const flce_params_t* p) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  if (p->N < 0 || p->H <= 0 || p->V <= 0) return FLCE_ERR_INVALID_ARG;
  if (p->H % 8 != 0) return FLCE_ERR_ALIGNMENT;  // 16-byte TMA row pitch
  if (p->N > (1LL << 30) || p->V > (1LL << 30) || p->H > (1LL << 20)) return FLCE_ERR_UNSUPPORTED;
  // Tile indices are int32 in the kernels: the 128 x 256 tile grid of x W^T
  // (and of the backward GEMMs, which are smaller) must stay below 2^31.
  if (((p->N + 127) / 128) * ((p->V + 255) / 256) >= (1LL << 31)) return FLCE_ERR_UNSUPPORTED;
  if (p->reduction < 0 || p->reduction > 2) return FLCE_ERR_INVALID_ARG;
  if (!(p->label_smoothing >= 0.f && p->label_smoothing <= 1.f)) return FLCE_ERR_INVALID_ARG;
  if (!(p->lse_square_scale >= 0.f) || !(p->lse_square_scale < INFINITY)) return FLCE_ERR_INVALID_ARG;
  if (!(p->logit_scale > -INFINITY && p->logit_scale < INFINITY)) return FLCE_ERR_INVALID_ARG;
  if (p->bwd_vocab_block < 0 || p->bwd_vocab_block % 256 != 0) return FLCE_ERR_INVALID_ARG;
  if (p->keep_vocab < 0 || p->keep_vocab % 256 != 0) return FLCE_ERR_INVALID_ARG;
  if (p->has_bias != 0 && p->has_bias != 1) return FLCE_ERR_INVALID_ARG;
  if (p->input_fp16 != 0 && p->input_fp16 != 1) return FLCE_ERR_INVALID_ARG;
  if (p->gemm_form < FLCE_GEMM_DEFAULT || p->gemm_form > FLCE_GEMM_WIDE_PAIR)
    return FLCE_ERR_INVALID_ARG;
  if (p->vocab_total == 0) {
    if (p->vocab_start != 0) return FLCE_ERR_INVALID_ARG;
  } else if (p->vocab_total < 0 || p->vocab_total > (1LL << 30) || p->vocab_start < 0 ||
             p->vocab_start + p->V > p->vocab_total) {
    return FLCE_ERR_INVALID_ARG;
  }
  return FLCE_OK;
}

// Full vocabulary size (the shard's own V when unsharded).
int64_t vocab_total(const flce_params_t* p) { return p->vocab_total > 0 ? p->vocab_total : p->V; }

// Plain (whole-vocabulary) calls: W must hold every vocabulary row.
bool whole_vocab(const flce_params_t* p) {
  return p->vocab_total == 0 || (p->vocab_total == p->V && p->vocab_start == 0);
}

struct Carver {
  uintptr_t base, cur, end;
  explicit Carver(void* b, size_t n)
      : base(reinterpret_cast<uintptr_t>(b)),
        cur((reinterpret_cast<uintptr_t>(b) + kAlign - 1) & ~(kAlign - 1)),
        end(reinterpret_cast<uintptr_t>(b) + n) {}
  template <class T>
  T* take(size_t count) {
    T* r = reinterpret_cast<T*>(cur);
    cur = (cur + count * sizeof(T) + kAlign - 1) & ~(kAlign - 1);
    return r;
  }
  size_t used() const { return cur - base; }
};

struct FwdWs {
  float *part_m, *part_d, *part_s, *zy;
  double* blk_sum;
  int* blk_cnt;
};

// The same carving serves sizing (base = null) and use.
size_t carve_fwd(const flce_params_t* p, void* base, FwdWs* w) {
  const size_t N = static_cast<size_t>(p->N);
  const size_t NT = static_cast<size_t>(cdiv(p->V, kBN));
  const size_t nblk = static_cast<size_t>(cdiv(p->N, kMergeRows));
  Carver c(base, 0);
  w->part_m = c.take<float>(NT * N);
  w->part_d = c.take<float>(NT * N);
  w->part_s = p->label_smoothing > 0.f ? c.take<float>(NT * N) : nullptr;
  w->zy = c.take<float>(N);
  w->blk_sum = c.take<double>(nblk);
  w->blk_cnt = c.take<int>(nblk);
  return c.used() + kAlign;  // slack for an unaligned base
}

int64_t vocab_block(const flce_params_t* p) {
  int64_t bv = p->bwd_vocab_block;
  if (bv <= 0) {
    const int64_t n = p->N > 0 ? p->N : 1;
    bv = kDlBudgetBytes / (n * 2) / 256 * 256;
    if (bv < kMinVocabBlock) bv = kMinVocabBlock;
  }
  const int64_t vr = (p->V + 255) / 256 * 256;
  return bv < vr ? bv : vr;
}

// Width of the kept block (the keep calls' first backward block): keep_vocab
// columns, at least BVc (0 = BVc), at most the vocabulary rounded up to 256.
int64_t kept_width(const flce_params_t* p) {
  const int64_t bv = vocab_block(p);
  const int64_t vr = (p->V + 255) / 256 * 256;
  const int64_t k = p->keep_vocab > bv ? p->keep_vocab : bv;
  return k < vr ? k : vr;
}

// Backward vocabulary blocks: [0, Vb0) is the kept block in the keep calls
// (kept_width wide) and the first BVc block otherwise; the rest follow in
// blocks of BVc, the last one ragged.
struct Blocks {
  int64_t first, bv;
  int count;
  Blocks(const flce_params_t* p, bool kept) : bv(vocab_block(p)) {
    first = std::min<int64_t>(kept ? kept_width(p) : bv, p->V);
    count = 1 + cdiv(p->V - first, bv);
  }
  int64_t start(int i) const { return i == 0 ? 0 : first + (i - 1) * bv; }
  int64_t width(int i, int64_t V) const {
    return i == 0 ? first : std::min<int64_t>(bv, V - start(i));
  }
};


struct BwdWs {
  float4* coef;
  uint16_t* dL;      // bf16 or fp16, like the operands
  float* dx_acc;
  float* db_part;
  float* dl_scale;   // [2]
};

// kept: the backward of a kept-block forward stages dL in the kept buffer,
// so its workspace holds no dL block; its db column partials are as wide as
// the kept block.
size_t carve_bwd(const flce_params_t* p, void* base, BwdWs* w, bool kept = false) {
  const size_t N = static_cast<size_t>(p->N);
  const int64_t bv = vocab_block(p);
  const Blocks blocks(p, kept);
  const int64_t db_cols = kept ? kept_width(p) : bv;
  Carver c(base, 0);
  w->coef = c.take<float4>(N);
  w->dl_scale = c.take<float>(2);
  w->dL = kept ? nullptr : c.take<uint16_t>(N * static_cast<size_t>(bv));
  w->dx_acc = blocks.count > 1 ? c.take<float>(N * static_cast<size_t>(p->H)) : nullptr;
  w->db_part = p->has_bias
                   ? c.take<float>(static_cast<size_t>(cdiv(p->N, kBM)) * 4 * db_cols)
                   : nullptr;
  return c.used() + kAlign;
}

// State kept between flce_forward_keep and flce_backward_keep: the kept
// block's q [N, ld] (ld = kept_width, cols = its columns inside the
// vocabulary; converted in place into the block's dL, then the staging buffer
// of the recomputed blocks) as fp16, then the running maxima of its 32-column
// chunks [ceil(cols / 32), N] fp32.
struct Kept {
  uint16_t* dq;
  float* kmax;
  int64_t ld;
  int cols;
};

size_t carve_kept(const flce_params_t* p, void* base, Kept* k) {
  const size_t N = static_cast<size_t>(p->N);
  const int64_t kw = kept_width(p);
  Carver c(base, 0);
  k->ld = kw;
  k->cols = static_cast<int>(kw < p->V ? kw : p->V);
  k->dq = c.take<uint16_t>(N * static_cast<size_t>(kw));
  k->kmax = c.take<float>(static_cast<size_t>(cdiv(k->cols, 32)) * N);
  return c.used() + kAlign;
}

// The stored-probability mode is the kept-block mode with one backward
// vocabulary block spanning the whole vocabulary: every probability is kept
// and nothing is recomputed.
flce_params_t whole_vocab_block(const flce_params_t* p) {
  flce_params_t q = *p;
  q.bwd_vocab_block = (p->V + 255) / 256 * 256;
  q.keep_vocab = 0;
  return q;
}

GemmGeom geom(int M, int N, int K, bool fp16) {
  GemmGeom g;
  std::memset(&g, 0, sizeof(g));
  g.ab_fp16 = fp16 ? 1 : 0;
  g.M = M;
  g.N = N;
  g.K = K;
  g.tiles_m = cdiv(M, kBM);
  g.tiles_n = cdiv(N, kBN);
  g.k_blocks = cdiv(K, kBK);
  g.raster_m_inner = 1;
  return g;
}

// Tile order. FLCE_RASTER=0 selects the plain orders (M inner for the
// logits GEMMs, N inner for dW / dx); the default bands the reused operand so
// its slice stays in L2 (bands of 16 pair-M-tiles = 4096 tokens of x for the
// logits GEMMs, 8 N-tiles = 2048 columns of x for dW).
bool use_bands() {
  const char* e = std::getenv("FLCE_RASTER");
  return !(e && e[0] == '0');
}

int grid_for(const GemmGeom& g, int sms) {
  const int tiles = g.tiles_m * g.tiles_n;
  return tiles < sms ? tiles : sms;
}

// NVTX range over a scope (host timeline; free unless a profiler is attached),
// so Nsight Systems shows each call and each backward vocabulary block.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Records the caller's events around each launch (flce_trace_t in flce.h).
struct Tracer {
  flce_trace_t* t;
  cudaStream_t s;
  bool begin() {
    if (!t) return true;
    t->count = 0;
    if (!t->events || t->capacity < 1) return true;
    if (cudaEventRecord(static_cast<cudaEvent_t>(t->events[0]), s) != cudaSuccess) return false;
    t->count = 1;
    return true;
  }
  bool after(flce_kernel_t kind) {
    if (!t || t->count == 0 || t->count >= t->capacity) return true;
    if (t->kinds) t->kinds[t->count - 1] = kind;
    if (cudaEventRecord(static_cast<cudaEvent_t>(t->events[t->count]), s) != cudaSuccess)
      return false;
    ++t->count;
    return true;
  }
};

}  // namespace

// kept: the kept block (flce_forward_keep / flce_backward_keep, and the
// stored mode with a block spanning the vocabulary); shard_stats / shard: the
// vocabulary-shard calls. NVTX names the call by `name`.
static flce_status_t forward_impl(const char* name, const flce_params_t* p, const void* x,
                                  const void* W, const void* b, const int64_t* y, float* loss,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_err, void* stream, flce_trace_t* trace,
                                  float* shard_stats = nullptr, void* kept = nullptr,
                                  size_t kept_bytes = 0);
static flce_status_t backward_impl(const char* name, const flce_params_t* p, const float* dloss,
                                   const float* lse, const void* x, const void* W, const void* b,
                                   const int64_t* y, void* dx, void* dW, void* db,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                   void* stream, flce_trace_t* trace, bool shard = false,
                                   void* kept = nullptr, size_t kept_bytes = 0);

extern "C" {

int32_t flce_resolved_gemm_form(const flce_params_t* p, int32_t which) {
  if (!p || which < 0 || which > 3 || check_params(p) != FLCE_OK) return -1;
  const int64_t N = p->N, H = p->H, V = p->V;
  const int64_t Vb = std::min<int64_t>(vocab_block(p), V);
  const GemmKind kind = gemm_kind(p);
  GemmKind k;
  switch (which) {
    case 0: k = gemm_for(kind, N, V, H); break;
    case 1: k = gemm_for(kind, N, Vb, H); break;
    case 2: k = gemm_for(kind, Vb, H, N); break;
    default: k = kind == kGemmSingle ? kGemmSingle : kGemmPair; break;  // dx
  }
  switch (k) {
    case kGemmSingle: return FLCE_GEMM_SINGLE_CTA;
    case kGemmWide: return FLCE_GEMM_WIDE_PAIR;
    default: return FLCE_GEMM_CTA_PAIR;
  }
}

size_t flce_workspace_size(const flce_params_t* p, int which) {
  if (check_params(p) != FLCE_OK || p->N == 0) return 0;
  if (which == 0) {
    FwdWs w;
    return carve_fwd(p, nullptr, &w);
  }
  if (which == 1 || which == 2) {
    BwdWs w;
    return carve_bwd(p, nullptr, &w, which == 2);
  }
  if (which == 3) {
    const flce_params_t q = whole_vocab_block(p);
    BwdWs w;
    return carve_bwd(&q, nullptr, &w, true);
  }
  return 0;
}

flce_status_t flce_forward(const flce_params_t* p, const void* x, const void* W, const void* b,
                           const int64_t* y, float* loss, float* lse, void* workspace,
                           size_t workspace_bytes, int32_t* dev_err, void* stream) {
  return flce_forward_traced(p, x, W, b, y, loss, lse, workspace, workspace_bytes, dev_err,
                             stream, nullptr);
}

flce_status_t flce_forward_traced(const flce_params_t* p, const void* x, const void* W,
                                  const void* b, const int64_t* y, float* loss, float* lse,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                  void* stream, flce_trace_t* trace) {
  return forward_impl("flce_forward", p, x, W, b, y, loss, lse, workspace, workspace_bytes,
                      dev_err, stream, trace);
}

flce_status_t flce_forward_store(const flce_params_t* p, const void* x, const void* W,
                                 const void* b, const int64_t* y, float* loss, float* lse,
                                 void* saved, size_t saved_bytes, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream,
                                 flce_trace_t* trace) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  if (!saved && p->N > 0) return FLCE_ERR_INVALID_ARG;
  const flce_params_t q = whole_vocab_block(p);
  return forward_impl("flce_forward_store", &q, x, W, b, y, loss, lse, workspace,
                      workspace_bytes, dev_err, stream, trace, nullptr, saved, saved_bytes);
}

size_t flce_saved_size(const flce_params_t* p) {
  if (check_params(p) != FLCE_OK || p->N == 0 || !whole_vocab(p)) return 0;
  const flce_params_t q = whole_vocab_block(p);
  Kept k{};
  return carve_kept(&q, nullptr, &k);
}

size_t flce_kept_size(const flce_params_t* p) {
  if (check_params(p) != FLCE_OK || p->N == 0) return 0;
  Kept k{};
  return carve_kept(p, nullptr, &k);
}

int64_t flce_keep_vocab_within(const flce_params_t* p, size_t extra_bytes) {
  if (check_params(p) != FLCE_OK || p->N == 0) return 0;
  BwdWs w;
  const size_t limit = carve_bwd(p, nullptr, &w, false) + extra_bytes;
  const int64_t bv = vocab_block(p);
  flce_params_t q = *p;
  for (int64_t k = 0; p->V - k * bv > bv; ++k) {
    q.keep_vocab = (p->V - k * bv + 255) / 256 * 256;
    Kept kk{};
    BwdWs wk;
    if (carve_kept(&q, nullptr, &kk) + carve_bwd(&q, nullptr, &wk, true) <= limit)
      return q.keep_vocab;
  }
  return bv;
}

flce_status_t flce_forward_keep(const flce_params_t* p, const void* x, const void* W,
                                const void* b, const int64_t* y, float* loss, float* lse,
                                void* kept, size_t kept_bytes, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err, void* stream,
                                flce_trace_t* trace) {
  if (!kept && p && p->N > 0) return FLCE_ERR_INVALID_ARG;
  return forward_impl("flce_forward_keep", p, x, W, b, y, loss, lse, workspace, workspace_bytes,
                      dev_err, stream, trace, nullptr, kept, kept_bytes);
}

}  // extern "C"

static flce_status_t forward_impl(const char* name, const flce_params_t* p, const void* x,
                                  const void* W, const void* b, const int64_t* y, float* loss,
                                  float* lse, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_err, void* stream, flce_trace_t* trace,
                                  float* shard_stats, void* kept, size_t kept_bytes) {
  NvtxRange nvtx_range(name);
  flce_status_t st = check_params(p);
  if (st != FLCE_OK) return st;
  if (shard_stats) {
    if (p->vocab_total == 0) return FLCE_ERR_INVALID_ARG;
    if (p->N == 0) return FLCE_OK;
  } else if (!whole_vocab(p) || !loss) {
    return FLCE_ERR_INVALID_ARG;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->N == 0) {
    if (p->reduction != FLCE_REDUCTION_NONE &&
        cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess)
      return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  if (!x || !W || !y || (!shard_stats && !lse) || !workspace || (p->has_bias && !b))
    return FLCE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W) || (p->has_bias && !aligned16(b))) return FLCE_ERR_ALIGNMENT;
  FwdWs w;
  const size_t need = carve_fwd(p, nullptr, &w);
  if (workspace_bytes < need) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  Kept kp{};  // filled by carve_kept when `kept` is given
  if (kept) {
    if (kept_bytes < carve_kept(p, nullptr, &kp)) return FLCE_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(kept)) return FLCE_ERR_ALIGNMENT;
  }
  int sms = 0;
  if ((st = device_info(&sms)) != FLCE_OK) return st;
  carve_fwd(p, workspace, &w);
  if (kept) carve_kept(p, kept, &kp);

  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  const GemmKind kind = gemm_for(gemm_kind(p), p->N, p->V, p->H);
  const bool pair = kind != kGemmSingle;
  CUtensorMap mx, mw;
  if (!encode_2d(&mx, x, H, N, static_cast<uint64_t>(H) * 2, kBK, kBM, p->input_fp16 != 0) ||
      !encode_2d(&mw, W, H, V, static_cast<uint64_t>(H) * 2, kBK, pair ? kBN / 2 : kBN,
                 p->input_fp16 != 0))
    return FLCE_ERR_CUDA;

  Tracer tr{trace, s};
  if (!tr.begin()) return FLCE_ERR_CUDA;
  const bool f16 = p->input_fp16 != 0;
  GemmGeom g = geom(N, V, H, f16);
  if (use_bands()) g.band_m = pair ? 16 : 32;
  FwdLseArgs ea;
  ea.bias = static_cast<const uint16_t*>(p->has_bias ? b : nullptr);
  ea.fp16 = f16 ? 1 : 0;
  ea.y = y;
  ea.y_off = p->vocab_start;
  ea.scale = p->logit_scale;
  ea.V = V;
  ea.Ntok = N;
  ea.part_m = w.part_m;
  ea.part_d = w.part_d;
  ea.part_s = w.part_s;
  ea.zy = w.zy;
  ea.keep_cols = 0;
  ea.keep_max = nullptr;
  std::memset(&ea.keep_map, 0, sizeof(ea.keep_map));
  if (kept) {
    ea.keep_cols = kp.cols;
    ea.keep_max = kp.kmax;
    if (!encode_store_2d(&ea.keep_map, kp.dq, kp.cols, N, static_cast<uint64_t>(kp.ld) * 2, false))
      return FLCE_ERR_CUDA;
  }
  const cudaError_t le =
      launch_fwd_lse(kind, mx, mw, g, ea, p->has_bias != 0, p->label_smoothing > 0.f,
                     kept != nullptr, reinterpret_cast<int*>(dev_err), grid_for(g, sms), s);
  if (le != cudaSuccess || !tr.after(FLCE_KERNEL_FWD_LSE)) return FLCE_ERR_CUDA;

  if (shard_stats) {
    ShardStatsArgs sa;
    sa.part_m = w.part_m;
    sa.part_d = w.part_d;
    sa.part_s = w.part_s;
    sa.zy = w.zy;
    sa.y = y;
    sa.N = N;
    sa.NT = g.tiles_n;
    sa.vocab_start = p->vocab_start;
    sa.V = V;
    sa.V_total = vocab_total(p);
    sa.ignore_index = p->ignore_index;
    sa.stats = shard_stats;
    sa.dev_err = reinterpret_cast<int*>(dev_err);
    if (p->label_smoothing <= 0.f &&
        cudaMemsetAsync(shard_stats + 3 * static_cast<size_t>(N), 0, sizeof(float) * N, s) !=
            cudaSuccess)
      return FLCE_ERR_CUDA;
    if (launch_shard_stats(sa, s) != cudaSuccess || !tr.after(FLCE_KERNEL_FWD_MERGE))
      return FLCE_ERR_CUDA;
    return FLCE_OK;
  }

  MergeArgs ma;
  ma.part_m = w.part_m;
  ma.part_d = w.part_d;
  ma.part_s = w.part_s;
  ma.zy = w.zy;
  ma.y = y;
  ma.N = N;
  ma.NT = g.tiles_n;
  ma.V = static_cast<int>(vocab_total(p));
  ma.ignore_index = p->ignore_index;
  ma.eps = p->label_smoothing;
  ma.lam = p->lse_square_scale;
  ma.reduction = p->reduction;
  ma.lse = lse;
  ma.loss = loss;
  ma.blk_sum = w.blk_sum;
  ma.blk_cnt = w.blk_cnt;
  ma.dev_err = reinterpret_cast<int*>(dev_err);
  if (launch_merge(ma, s) != cudaSuccess || !tr.after(FLCE_KERNEL_FWD_MERGE)) return FLCE_ERR_CUDA;
  if (p->reduction != FLCE_REDUCTION_NONE &&
      (launch_finalize(ma, s) != cudaSuccess || !tr.after(FLCE_KERNEL_FWD_FINALIZE)))
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

extern "C" flce_status_t flce_backward(const flce_params_t* p, const float* dloss, const float* lse,
                            const void* x, const void* W, const void* b, const int64_t* y,
                            void* dx, void* dW, void* db, void* workspace, size_t workspace_bytes,
                            int32_t* dev_err, void* stream) {
  return flce_backward_traced(p, dloss, lse, x, W, b, y, dx, dW, db, workspace, workspace_bytes,
                              dev_err, stream, nullptr);
}

extern "C" flce_status_t flce_backward_traced(const flce_params_t* p, const float* dloss,
                                              const float* lse, const void* x, const void* W,
                                              const void* b, const int64_t* y, void* dx, void* dW,
                                              void* db, void* workspace, size_t workspace_bytes,
                                              int32_t* dev_err, void* stream,
                                              flce_trace_t* trace) {
  return backward_impl("flce_backward", p, dloss, lse, x, W, b, y, dx, dW, db, workspace,
                       workspace_bytes, dev_err, stream, trace);
}

extern "C" flce_status_t flce_backward_keep(const flce_params_t* p, const float* dloss,
                                            const float* lse, void* kept, size_t kept_bytes,
                                            const void* x, const void* W, const void* b,
                                            const int64_t* y, void* dx, void* dW, void* db,
                                            void* workspace, size_t workspace_bytes,
                                            int32_t* dev_err, void* stream, flce_trace_t* trace) {
  if (!kept && p && p->N > 0) return FLCE_ERR_INVALID_ARG;
  return backward_impl("flce_backward_keep", p, dloss, lse, x, W, b, y, dx, dW, db, workspace,
                       workspace_bytes, dev_err, stream, trace, false, kept, kept_bytes);
}

extern "C" flce_status_t flce_backward_store(const flce_params_t* p, const float* dloss,
                                             const float* lse, void* saved, size_t saved_bytes,
                                             const void* x, const void* W, const void* b,
                                             const int64_t* y, void* dx, void* dW, void* db,
                                             void* workspace, size_t workspace_bytes,
                                             int32_t* dev_err, void* stream,
                                             flce_trace_t* trace) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  if (!saved && p->N > 0) return FLCE_ERR_INVALID_ARG;
  const flce_params_t q = whole_vocab_block(p);
  return backward_impl("flce_backward_store", &q, dloss, lse, x, W, b, y, dx, dW, db, workspace,
                       workspace_bytes, dev_err, stream, trace, false, saved, saved_bytes);
}

static flce_status_t backward_impl(const char* name, const flce_params_t* p, const float* dloss,
                                   const float* lse, const void* x, const void* W, const void* b,
                                   const int64_t* y, void* dx, void* dW, void* db,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                   void* stream, flce_trace_t* trace, bool shard, void* kept,
                                   size_t kept_bytes) {
  NvtxRange nvtx_range(name);
  flce_status_t st = check_params(p);
  if (st != FLCE_OK) return st;
  if (shard ? p->vocab_total == 0 : !whole_vocab(p)) return FLCE_ERR_INVALID_ARG;
  if (!dW || (p->has_bias && !db)) return FLCE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t dw_bytes = static_cast<size_t>(p->V) * p->H * (p->dW_fp32 ? 4 : 2);
  if (p->N == 0) {
    if (cudaMemsetAsync(dW, 0, dw_bytes, s) != cudaSuccess) return FLCE_ERR_CUDA;
    if (p->has_bias &&
        cudaMemsetAsync(db, 0, static_cast<size_t>(p->V) * (p->db_fp32 ? 4 : 2), s) != cudaSuccess)
      return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  if (!dloss || !lse || !x || !W || !y || !dx || !workspace || (p->has_bias && !b))
    return FLCE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W) || (p->has_bias && !aligned16(b)) || !aligned16(dx) ||
      !aligned16(dW))
    return FLCE_ERR_ALIGNMENT;
  BwdWs w;
  const size_t need = carve_bwd(p, nullptr, &w, kept != nullptr);
  if (workspace_bytes < need) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  Kept kp{};  // filled by carve_kept when `kept` is given
  if (kept) {
    if (kept_bytes < carve_kept(p, nullptr, &kp)) return FLCE_ERR_WORKSPACE_TOO_SMALL;
    if (!aligned16(kept)) return FLCE_ERR_ALIGNMENT;
    carve_kept(p, kept, &kp);
  }
  int sms = 0;
  if ((st = device_info(&sms)) != FLCE_OK) return st;
  carve_bwd(p, workspace, &w, kept != nullptr);
  // The kept buffer is every block's dL staging buffer: the kept block's own
  // [N, ld] array, then [N, BVc] blocks at its start.
  if (kept) w.dL = kp.dq;

  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  const Blocks blocks(p, kept != nullptr);
  const int64_t bv = blocks.bv;
  const int nblk = blocks.count;
  const int ld_db = static_cast<int>(kept ? kp.ld : bv);
  int* derr = reinterpret_cast<int*>(dev_err);
  const GemmKind kind = gemm_kind(p);
  const bool pair = kind != kGemmSingle;

  Tracer tr{trace, s};
  if (!tr.begin()) return FLCE_ERR_CUDA;
  PrepArgs pa;
  pa.dloss = dloss;
  pa.lse = lse;
  pa.y = y;
  pa.N = N;
  pa.ignore_index = p->ignore_index;
  pa.V = static_cast<int>(vocab_total(p));
  pa.eps = p->label_smoothing;
  pa.lam = p->lse_square_scale;
  pa.scale = p->logit_scale;
  pa.reduction = p->reduction;
  pa.coef = w.coef;
  pa.fp16 = p->input_fp16;
  pa.dl_scale = w.dl_scale;
  pa.dev_err = derr;
  if (launch_prep(pa, s) != cudaSuccess || !tr.after(FLCE_KERNEL_BWD_PREP)) return FLCE_ERR_CUDA;

  const bool f16 = p->input_fp16 != 0;
  CUtensorMap mx_k, mw_k, mx_mn, mw_mn;
  if (!encode_2d(&mx_k, x, H, N, static_cast<uint64_t>(H) * 2, kBK, kBM, f16) ||
      !encode_2d(&mw_k, W, H, V, static_cast<uint64_t>(H) * 2, kBK, pair ? kBN / 2 : kBN, f16) ||
      !encode_2d(&mx_mn, x, H, N, static_cast<uint64_t>(H) * 2, 64, kBK, f16) ||
      !encode_2d(&mw_mn, W, H, V, static_cast<uint64_t>(H) * 2, 64, kBK, f16))
    return FLCE_ERR_CUDA;

  for (int blk = 0; blk < nblk; ++blk) {
    NvtxRange nvtx_block("flce_backward_vocab_block");
    const int v0 = static_cast<int>(blocks.start(blk));
    const int Vb = static_cast<int>(blocks.width(blk, V));
    const bool from_kept = kept && blk == 0;
    // Row pitch (elements) of this block's dL.
    const int64_t ld = from_kept ? kp.ld : bv;
    CUtensorMap mdl_k, mdl_mn;
    if (!encode_2d(&mdl_k, w.dL, Vb, N, static_cast<uint64_t>(ld) * 2, kBK, kBM, f16) ||
        !encode_2d(&mdl_mn, w.dL, Vb, N, static_cast<uint64_t>(ld) * 2, 64, kBK, f16))
      return FLCE_ERR_CUDA;

    // Recompute the block's logits (or, for the kept block, read the kept
    // probabilities) and form dL (bf16) and db partials.
    int db_parts = 0;
    if (from_kept) {
      // In place: the kept q of block 0 becomes its dL.
      ConvertArgs ca;
      ca.q = reinterpret_cast<const __half*>(kp.dq);
      ca.ld_q = static_cast<int>(kp.ld);
      ca.chunk_max = kp.kmax;
      ca.coef = w.coef;
      ca.y = y;
      ca.y_off = p->vocab_start;
      ca.N = N;
      ca.v0 = 0;
      ca.Vb = Vb;
      ca.dL = w.dL;
      ca.ld_dL = static_cast<int>(ld);
      ca.fp16 = p->input_fp16;
      ca.dl_scale = w.dl_scale;
      ca.db_part = w.db_part;
      ca.ld_db = ld_db;
      if (launch_convert(ca, s) != cudaSuccess || !tr.after(FLCE_KERNEL_BWD_CONVERT))
        return FLCE_ERR_CUDA;
      db_parts = convert_db_parts(N);
    }
    GemmGeom g1 = geom(N, Vb, H, f16);
    g1.b_mn_off = v0;
    if (use_bands()) g1.band_m = pair ? 16 : 32;
    DlogitsArgs da;
    da.bias = static_cast<const uint16_t*>(p->has_bias ? b : nullptr);
    da.fp16 = p->input_fp16;
    da.dl_scale = w.dl_scale;
    da.y = y;
    da.y_off = p->vocab_start;
    da.coef = w.coef;
    da.scale = p->logit_scale;
    da.V = V;
    da.Ntok = N;
    da.v0 = v0;
    da.Vb = Vb;
    da.db_part = w.db_part;
    da.ld_db = ld_db;
    if (!encode_store_2d(&da.dl_map, w.dL, Vb, N, static_cast<uint64_t>(ld) * 2, false))
      return FLCE_ERR_CUDA;
    if (!from_kept) {
      if (launch_dlogits(gemm_for(kind, N, Vb, H), mx_k, mw_k, g1, da, p->has_bias != 0, derr,
                         grid_for(g1, sms),
                         s) != cudaSuccess ||
          !tr.after(FLCE_KERNEL_BWD_DLOGITS))
        return FLCE_ERR_CUDA;
      db_parts = g1.tiles_m * 4;
    }
    if (p->has_bias &&
        (launch_db_finalize(w.db_part, db_parts, ld_db, v0, Vb, db,
                            p->db_fp32 != 0, f16, s) != cudaSuccess ||
         !tr.after(FLCE_KERNEL_BWD_DB)))
      return FLCE_ERR_CUDA;

    // dW block: one GEMM over all tokens (M = vocab rows, K = tokens).
    GemmGeom g2 = geom(Vb, H, N, f16);
    g2.raster_m_inner = 0;
    const GemmKind k2 = gemm_for(kind, Vb, H, N);
    if (use_bands()) g2.band_n = k2 == kGemmWide ? 4 : 8;  // 2048 columns of x
    DwArgs wa;
    const size_t dw_elt = p->dW_fp32 ? 4 : 2;
    if (!encode_store_2d(&wa.out_map,
                         static_cast<char*>(dW) + static_cast<size_t>(v0) * H * dw_elt, H, Vb,
                         static_cast<uint64_t>(H) * dw_elt, p->dW_fp32 != 0))
      return FLCE_ERR_CUDA;
    wa.out_bf16 = p->dW_fp32 ? 0 : 1;
    wa.fp16 = p->input_fp16;
    wa.acc_scale = w.dl_scale + 1;
    wa.Mrows = Vb;
    wa.Ncols = H;
    if (launch_dw(k2, mdl_mn, mx_mn, g2, wa, derr, grid_for(g2, sms), s) != cudaSuccess ||
        !tr.after(FLCE_KERNEL_BWD_DW))
      return FLCE_ERR_CUDA;

    // dx += dL_blk W_blk (K = the block's vocab rows).
    GemmGeom g3 = geom(N, H, Vb, f16);
    g3.b_k_off = v0;
    g3.raster_m_inner = 0;
    DxArgs xa;
    xa.acc = w.dx_acc;
    xa.out = static_cast<uint16_t*>(dx);
    xa.out_f32 = shard ? 1 : 0;
    xa.fp16 = p->input_fp16;
    xa.acc_scale = w.dl_scale + 1;
    xa.ld = H;
    xa.Ntok = N;
    xa.Ncols = H;
    xa.first = blk == 0;
    xa.last = blk == nblk - 1;
    if (launch_dx(kind == kGemmSingle ? kGemmSingle : kGemmPair, mdl_k, mw_mn, g3, xa, derr,
                  grid_for(g3, sms), s) != cudaSuccess ||
        !tr.after(FLCE_KERNEL_BWD_DX))
      return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
}

extern "C" {

flce_status_t flce_forward_shard(const flce_params_t* p, const void* x, const void* W,
                                 const void* b, const int64_t* y, float* stats, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream) {
  if (!stats && p && p->N > 0) return FLCE_ERR_INVALID_ARG;
  return forward_impl("flce_forward_shard", p, x, W, b, y, nullptr, nullptr, workspace,
                      workspace_bytes, dev_err, stream, nullptr, stats);
}

flce_status_t flce_forward_shard_keep(const flce_params_t* p, const void* x, const void* W,
                                      const void* b, const int64_t* y, float* stats, void* kept,
                                      size_t kept_bytes, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_err, void* stream) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  if ((!stats || !kept) && p->N > 0) return FLCE_ERR_INVALID_ARG;
  return forward_impl("flce_forward_shard_keep", p, x, W, b, y, nullptr, nullptr, workspace,
                      workspace_bytes, dev_err, stream, nullptr, stats, kept, kept_bytes);
}

flce_status_t flce_shard_rescale(const flce_params_t* p, float* stats, const float* global_max,
                                 void* stream) {
  flce_status_t st = check_params(p);
  if (st != FLCE_OK) return st;
  if (p->N == 0) return FLCE_OK;
  if (!stats || !global_max) return FLCE_ERR_INVALID_ARG;
  return launch_shard_rescale(stats, global_max, static_cast<int>(p->N),
                              static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FLCE_OK
             : FLCE_ERR_CUDA;
}

flce_status_t flce_loss_from_stats(const flce_params_t* p, const float* stats, const int64_t* y,
                                   float* loss, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, void* stream) {
  flce_status_t st = check_params(p);
  if (st != FLCE_OK) return st;
  if (!loss) return FLCE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int N = static_cast<int>(p->N);
  if (N == 0) {
    if (p->reduction != FLCE_REDUCTION_NONE &&
        cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess)
      return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  if (!stats || !y || !lse || !workspace) return FLCE_ERR_INVALID_ARG;
  const int nblk = cdiv(N, kMergeRows);
  Carver c(workspace, 0);
  double* blk_sum = c.take<double>(nblk);
  int* blk_cnt = c.take<int>(nblk);
  if (workspace_bytes < c.used()) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  MergeArgs ma;
  ma.part_m = stats;
  ma.part_d = stats + N;
  ma.zy = stats + 2 * static_cast<size_t>(N);
  ma.part_s = p->label_smoothing > 0.f ? stats + 3 * static_cast<size_t>(N) : nullptr;
  ma.y = y;
  ma.N = N;
  ma.NT = 1;
  ma.V = static_cast<int>(vocab_total(p));
  ma.ignore_index = p->ignore_index;
  ma.eps = p->label_smoothing;
  ma.lam = p->lse_square_scale;
  ma.reduction = p->reduction;
  ma.lse = lse;
  ma.loss = loss;
  ma.blk_sum = blk_sum;
  ma.blk_cnt = blk_cnt;
  ma.dev_err = reinterpret_cast<int*>(dev_err);
  if (launch_merge(ma, s) != cudaSuccess) return FLCE_ERR_CUDA;
  if (p->reduction != FLCE_REDUCTION_NONE && launch_finalize(ma, s) != cudaSuccess)
    return FLCE_ERR_CUDA;
  return FLCE_OK;
}

flce_status_t flce_backward_shard(const flce_params_t* p, const float* dloss, const float* lse,
                                  const void* x, const void* W, const void* b, const int64_t* y,
                                  float* dx_partial, void* dW, void* db, void* workspace,
                                  size_t workspace_bytes, int32_t* dev_err, void* stream) {
  return backward_impl("flce_backward_shard", p, dloss, lse, x, W, b, y, dx_partial, dW, db,
                       workspace, workspace_bytes, dev_err, stream, nullptr, true);
}

flce_status_t flce_backward_shard_keep(const flce_params_t* p, const float* dloss,
                                       const float* lse, void* kept, size_t kept_bytes,
                                       const void* x, const void* W, const void* b,
                                       const int64_t* y, float* dx_partial, void* dW, void* db,
                                       void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                       void* stream) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  if (!kept && p->N > 0) return FLCE_ERR_INVALID_ARG;
  return backward_impl("flce_backward_shard_keep", p, dloss, lse, x, W, b, y, dx_partial, dW, db,
                       workspace, workspace_bytes, dev_err, stream, nullptr, true, kept,
                       kept_bytes);
}

flce_status_t flce_cast_f32(const float* src, void* dst, int64_t n, int32_t dst_fp16,
                            void* stream) {
  if (n < 0 || (n > 0 && (!src || !dst)) || (dst_fp16 != 0 && dst_fp16 != 1))
    return FLCE_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(dst)) return FLCE_ERR_ALIGNMENT;
  return launch_cast16(src, static_cast<uint16_t*>(dst), n, dst_fp16 != 0,
                       static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FLCE_OK
             : FLCE_ERR_CUDA;
}

flce_status_t flce_selftest_wait_timeout(int32_t* dev_err, int64_t limit_cycles, void* stream) {
  if (!dev_err || limit_cycles <= 0 || limit_cycles > (1LL << 32)) return FLCE_ERR_INVALID_ARG;
  int sms = 0;
  flce_status_t st = device_info(&sms);
  if (st != FLCE_OK) return st;
  return launch_wait_timeout_selftest(reinterpret_cast<int*>(dev_err), limit_cycles,
                                      static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FLCE_OK
             : FLCE_ERR_CUDA;
}

flce_status_t flce_read_device_error(int32_t* dev_err, void* stream, int32_t* host_err) {
  if (!dev_err) return FLCE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, dev_err, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return FLCE_ERR_CUDA;
  if (h != 0 && (cudaMemsetAsync(dev_err, 0, sizeof(int32_t), s) != cudaSuccess ||
                 cudaStreamSynchronize(s) != cudaSuccess))
    return FLCE_ERR_CUDA;
  if (host_err) *host_err = h;
  if (h & FLCE_DEVERR_TIMEOUT) return FLCE_ERR_TIMEOUT;
  if (h & FLCE_DEVERR_TARGET) return FLCE_ERR_TARGET_OUT_OF_RANGE;
  return FLCE_OK;
}

const char* flce_status_string(flce_status_t status) {
  switch (status) {
    case FLCE_OK: return "ok";
    case FLCE_ERR_INVALID_ARG: return "invalid argument";
    case FLCE_ERR_ALIGNMENT: return "alignment: H must be a multiple of 8 and x, W, b, dx, dW 16-byte aligned";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FLCE_ERR_TARGET_OUT_OF_RANGE: return "a target is outside [0, V) and not ignore_index";
    case FLCE_ERR_CUDA: return "CUDA runtime error";
    case FLCE_ERR_TIMEOUT: return "a kernel pipeline wait timed out";
    case FLCE_ERR_UNSUPPORTED: return "unsupported device (needs sm_103) or size";
  }
  return "unknown status";
}

const char* flce_version(void) { return "0.1.0"; }

}  // extern "C"
