// C ABI of the FLCE library (declared in include/flce.h): argument checks,
// workspace carving, TMA descriptor encoding and the launch sequence.
//
// Forward  (DeepSpeed PR #8792 "What": forward keeps per-token softmax
//           statistics only):
//   fwd_lse GEMM  x W^T tile by tile -> (m, d[, sum z]) partials + z_y
//   merge         partials -> lse, per-token loss, reduction
// Backward (same page: logits recomputed one vocabulary block at a time, so
//           each dW block is one GEMM over all tokens):
//   prep          per-token coefficients from dloss, lse, y
//   per vocab block [v0, v0 + Vb):
//     dlogits GEMM  recompute x W_blk^T -> dL_blk = s dz (bf16) + db partials
//     dW GEMM       dW[v0:v0+Vb] = dL_blk^T x            (K = all tokens)
//     dx GEMM       dx (+)= dL_blk W_blk                  (fp32 across blocks)
//     db finalize   (with a bias)
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/flce.h"
#include "epilogues.cuh"
#include "flce_internal.h"

using namespace flce;

namespace {

constexpr int64_t kDefaultVocabBlock = 16384;
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

// 2-D bf16 tensor [outer, inner] with row pitch `pitch_bytes`, 128-B swizzled
// boxes of box_inner x box_outer elements; out-of-range elements read as 0.
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer,
               uint64_t pitch_bytes, uint32_t box_inner, uint32_t box_outer) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {pitch_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int cdiv(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// GEMM kernel form: CTA pairs (cta_group::2, 256 x 256 tiles) or single CTAs
// (128 x 256 tiles). FLCE_CTA_PAIR=0 / 1 in the environment overrides the
// default; both forms compute identical results up to accumulation order.
bool use_cta_pair() {
  const char* e = std::getenv("FLCE_CTA_PAIR");
  if (e && e[0] == '0') return false;
  if (e && e[0] == '1') return true;
  return true;
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
  if (p->reduction < 0 || p->reduction > 2) return FLCE_ERR_INVALID_ARG;
  if (!(p->label_smoothing >= 0.f && p->label_smoothing <= 1.f)) return FLCE_ERR_INVALID_ARG;
  if (!(p->lse_square_scale >= 0.f) || !(p->lse_square_scale < INFINITY)) return FLCE_ERR_INVALID_ARG;
  if (!(p->logit_scale > -INFINITY && p->logit_scale < INFINITY)) return FLCE_ERR_INVALID_ARG;
  if (p->bwd_vocab_block < 0 || p->bwd_vocab_block % 256 != 0) return FLCE_ERR_INVALID_ARG;
  if (p->has_bias != 0 && p->has_bias != 1) return FLCE_ERR_INVALID_ARG;
  return FLCE_OK;
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
  const size_t nblk = static_cast<size_t>(cdiv(p->N, kMergeThreads));
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
  int64_t bv = p->bwd_vocab_block > 0 ? p->bwd_vocab_block : kDefaultVocabBlock;
  const int64_t vr = (p->V + 255) / 256 * 256;
  return bv < vr ? bv : vr;
}

struct BwdWs {
  float4* coef;
  __nv_bfloat16* dL;
  float* dx_acc;
  float* db_part;
};

size_t carve_bwd(const flce_params_t* p, void* base, BwdWs* w) {
  const size_t N = static_cast<size_t>(p->N);
  const int64_t bv = vocab_block(p);
  const int nblk = cdiv(p->V, bv);
  Carver c(base, 0);
  w->coef = c.take<float4>(N);
  w->dL = c.take<__nv_bfloat16>(N * static_cast<size_t>(bv));
  w->dx_acc = nblk > 1 ? c.take<float>(N * static_cast<size_t>(p->H)) : nullptr;
  w->db_part = p->has_bias ? c.take<float>(static_cast<size_t>(cdiv(p->N, kBM)) * 4 * bv) : nullptr;
  return c.used() + kAlign;
}

GemmGeom geom(int M, int N, int K) {
  GemmGeom g;
  std::memset(&g, 0, sizeof(g));
  g.M = M;
  g.N = N;
  g.K = K;
  g.tiles_m = cdiv(M, kBM);
  g.tiles_n = cdiv(N, kBN);
  g.k_blocks = cdiv(K, kBK);
  g.raster_m_inner = 1;
  return g;
}

int grid_for(const GemmGeom& g, int sms) {
  const int tiles = g.tiles_m * g.tiles_n;
  return tiles < sms ? tiles : sms;
}

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

extern "C" {

size_t flce_workspace_size(const flce_params_t* p, int which) {
  if (check_params(p) != FLCE_OK || p->N == 0) return 0;
  if (which == 0) {
    FwdWs w;
    return carve_fwd(p, nullptr, &w);
  }
  if (which == 1) {
    BwdWs w;
    return carve_bwd(p, nullptr, &w);
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
  flce_status_t st = check_params(p);
  if (st != FLCE_OK) return st;
  if (!loss) return FLCE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (p->N == 0) {
    if (p->reduction != FLCE_REDUCTION_NONE &&
        cudaMemsetAsync(loss, 0, sizeof(float), s) != cudaSuccess)
      return FLCE_ERR_CUDA;
    return FLCE_OK;
  }
  if (!x || !W || !y || !lse || !workspace || (p->has_bias && !b)) return FLCE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(W) || (p->has_bias && !aligned16(b))) return FLCE_ERR_ALIGNMENT;
  FwdWs w;
  const size_t need = carve_fwd(p, nullptr, &w);
  if (workspace_bytes < need) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0;
  if ((st = device_info(&sms)) != FLCE_OK) return st;
  carve_fwd(p, workspace, &w);

  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  const bool pair = use_cta_pair();
  CUtensorMap mx, mw;
  if (!encode_2d(&mx, x, H, N, static_cast<uint64_t>(H) * 2, kBK, kBM) ||
      !encode_2d(&mw, W, H, V, static_cast<uint64_t>(H) * 2, kBK, pair ? kBN / 2 : kBN))
    return FLCE_ERR_CUDA;

  Tracer tr{trace, s};
  if (!tr.begin()) return FLCE_ERR_CUDA;
  GemmGeom g = geom(N, V, H);
  FwdLseArgs ea;
  ea.bias = static_cast<const __nv_bfloat16*>(p->has_bias ? b : nullptr);
  ea.y = y;
  ea.scale = p->logit_scale;
  ea.V = V;
  ea.Ntok = N;
  ea.part_m = w.part_m;
  ea.part_d = w.part_d;
  ea.part_s = w.part_s;
  ea.zy = w.zy;
  if (launch_fwd_lse(pair, mx, mw, g, ea, p->has_bias != 0, p->label_smoothing > 0.f,
                     reinterpret_cast<int*>(dev_err), grid_for(g, sms), s) != cudaSuccess ||
      !tr.after(FLCE_KERNEL_FWD_LSE))
    return FLCE_ERR_CUDA;

  MergeArgs ma;
  ma.part_m = w.part_m;
  ma.part_d = w.part_d;
  ma.part_s = w.part_s;
  ma.zy = w.zy;
  ma.y = y;
  ma.N = N;
  ma.NT = g.tiles_n;
  ma.V = V;
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

flce_status_t flce_backward(const flce_params_t* p, const float* dloss, const float* lse,
                            const void* x, const void* W, const void* b, const int64_t* y,
                            void* dx, void* dW, void* db, void* workspace, size_t workspace_bytes,
                            int32_t* dev_err, void* stream) {
  return flce_backward_traced(p, dloss, lse, x, W, b, y, dx, dW, db, workspace, workspace_bytes,
                              dev_err, stream, nullptr);
}

flce_status_t flce_backward_traced(const flce_params_t* p, const float* dloss, const float* lse,
                                   const void* x, const void* W, const void* b, const int64_t* y,
                                   void* dx, void* dW, void* db, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, void* stream,
                                   flce_trace_t* trace) {
  flce_status_t st = check_params(p);
  if (st != FLCE_OK) return st;
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
  const size_t need = carve_bwd(p, nullptr, &w);
  if (workspace_bytes < need) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0;
  if ((st = device_info(&sms)) != FLCE_OK) return st;
  carve_bwd(p, workspace, &w);

  const int N = static_cast<int>(p->N), H = static_cast<int>(p->H), V = static_cast<int>(p->V);
  const int64_t bv = vocab_block(p);
  const int nblk = cdiv(V, bv);
  int* derr = reinterpret_cast<int*>(dev_err);
  const bool pair = use_cta_pair();

  Tracer tr{trace, s};
  if (!tr.begin()) return FLCE_ERR_CUDA;
  PrepArgs pa;
  pa.dloss = dloss;
  pa.lse = lse;
  pa.y = y;
  pa.N = N;
  pa.V = V;
  pa.ignore_index = p->ignore_index;
  pa.eps = p->label_smoothing;
  pa.lam = p->lse_square_scale;
  pa.scale = p->logit_scale;
  pa.reduction = p->reduction;
  pa.coef = w.coef;
  pa.dev_err = derr;
  if (launch_prep(pa, s) != cudaSuccess || !tr.after(FLCE_KERNEL_BWD_PREP)) return FLCE_ERR_CUDA;

  CUtensorMap mx_k, mw_k, mx_mn, mw_mn;
  if (!encode_2d(&mx_k, x, H, N, static_cast<uint64_t>(H) * 2, kBK, kBM) ||
      !encode_2d(&mw_k, W, H, V, static_cast<uint64_t>(H) * 2, kBK, pair ? kBN / 2 : kBN) ||
      !encode_2d(&mx_mn, x, H, N, static_cast<uint64_t>(H) * 2, 64, kBK) ||
      !encode_2d(&mw_mn, W, H, V, static_cast<uint64_t>(H) * 2, 64, kBK))
    return FLCE_ERR_CUDA;

  for (int blk = 0; blk < nblk; ++blk) {
    const int v0 = static_cast<int>(blk * bv);
    const int Vb = static_cast<int>(V - v0 < bv ? V - v0 : bv);
    CUtensorMap mdl_k, mdl_mn;
    if (!encode_2d(&mdl_k, w.dL, Vb, N, static_cast<uint64_t>(bv) * 2, kBK, kBM) ||
        !encode_2d(&mdl_mn, w.dL, Vb, N, static_cast<uint64_t>(bv) * 2, 64, kBK))
      return FLCE_ERR_CUDA;

    // Recompute the block's logits and form dL (bf16) and db partials.
    GemmGeom g1 = geom(N, Vb, H);
    g1.b_mn_off = v0;
    DlogitsArgs da;
    da.bias = static_cast<const __nv_bfloat16*>(p->has_bias ? b : nullptr);
    da.y = y;
    da.coef = w.coef;
    da.scale = p->logit_scale;
    da.V = V;
    da.Ntok = N;
    da.v0 = v0;
    da.Vb = Vb;
    da.dL = w.dL;
    da.ld_dL = static_cast<int>(bv);
    da.db_part = w.db_part;
    da.ld_db = static_cast<int>(bv);
    if (launch_dlogits(pair, mx_k, mw_k, g1, da, p->has_bias != 0, derr, grid_for(g1, sms), s) !=
            cudaSuccess ||
        !tr.after(FLCE_KERNEL_BWD_DLOGITS))
      return FLCE_ERR_CUDA;
    if (p->has_bias &&
        (launch_db_finalize(w.db_part, g1.tiles_m * 4, static_cast<int>(bv), v0, Vb, db,
                            p->db_fp32 != 0, s) != cudaSuccess ||
         !tr.after(FLCE_KERNEL_BWD_DB)))
      return FLCE_ERR_CUDA;

    // dW block: one GEMM over all tokens (M = vocab rows, K = tokens).
    GemmGeom g2 = geom(Vb, H, N);
    g2.raster_m_inner = 0;
    DwArgs wa;
    wa.out = dW;
    wa.out_bf16 = p->dW_fp32 ? 0 : 1;
    wa.ld = H;
    wa.row0 = v0;
    wa.Mrows = Vb;
    wa.Ncols = H;
    if (launch_dw(pair, mdl_mn, mx_mn, g2, wa, derr, grid_for(g2, sms), s) != cudaSuccess ||
        !tr.after(FLCE_KERNEL_BWD_DW))
      return FLCE_ERR_CUDA;

    // dx += dL_blk W_blk (K = the block's vocab rows).
    GemmGeom g3 = geom(N, H, Vb);
    g3.b_k_off = v0;
    g3.raster_m_inner = 0;
    DxArgs xa;
    xa.acc = w.dx_acc;
    xa.out = static_cast<__nv_bfloat16*>(dx);
    xa.ld = H;
    xa.Ntok = N;
    xa.Ncols = H;
    xa.first = blk == 0;
    xa.last = blk == nblk - 1;
    if (launch_dx(pair, mdl_k, mw_mn, g3, xa, derr, grid_for(g3, sms), s) != cudaSuccess ||
        !tr.after(FLCE_KERNEL_BWD_DX))
      return FLCE_ERR_CUDA;
  }
  return FLCE_OK;
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
