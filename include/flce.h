/*
 * flce.h - C ABI of the GB300 (sm_103a) fused linear cross-entropy library.
 *
 * Fused linear cross-entropy (FLCE) computes the loss of a final linear
 * layer followed by cross-entropy without ever holding the [N, V] logits:
 *
 *   z[n, v]  = s * (x[n, :] . W[v, :] + b[v])
 *   lse[n]   = log sum_v exp(z[n, v])
 *   l[n]     = (1 - eps)(lse[n] - z[n, y_n]) + eps * lse[n]
 *              - (eps / V) sum_v z[n, v] + lam * lse[n]^2      (0 if y_n == ignore_index)
 *   loss     = l (none) | sum_n l[n] (sum) | sum_n l[n] / total (mean)
 *
 * and, in the backward pass, with g[n] the upstream gradient of token n's loss
 * (dloss, dloss / total or dloss[n]; 0 for ignored tokens) and p = exp(z - lse):
 *
 *   dz[n, v] = g[n] * ((1 + 2 lam lse[n]) p[n, v] - eps / V - (1 - eps) [v == y_n])
 *   dx = s dz W,   dW = s dz^T x,   db = s sum_n dz[n, :]
 *
 * Sources: the loss, label smoothing, logit_scale, ignore_index and the
 * "mean over non-ignored tokens" rule follow the flash-linear-attention module
 * fla/modules/fused_linear_cross_entropy.py (cross_entropy_kernel and
 * fused_linear_cross_entropy_forward); the z-loss lam * lse^2 and the gradient
 * (1 + 2 lam lse) softmax - eps/V - (1 - eps) delta follow Liger-Kernel PR #239
 * "Support Z Loss in CE" (Details); reduction "none" and the "forward keeps
 * only per-token softmax statistics, backward recomputes the logits one
 * vocabulary block at a time" structure follow DeepSpeed PR #8792 ("What").
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers on the current CUDA device,
 *    except where a parameter says HOST. Tensors are dense and row-major.
 *  - The caller owns every buffer, the workspace included. The library never
 *    allocates or frees device memory and keeps no per-call state; calls are
 *    stream-ordered on `stream` (a cudaStream_t; NULL = legacy default stream)
 *    and return without synchronising.
 *  - Host-detectable errors (bad sizes, null or misaligned pointers, a small
 *    workspace) return a status before anything is launched. Errors only the
 *    device can see (an out-of-range target, a pipeline wait that timed out)
 *    are OR-ed into the caller's device word `dev_err` (FLCE_DEVERR_* bits);
 *    read it with flce_read_device_error after the stream has run. Outputs of
 *    a call that raised a device error are unspecified. Kernels never trap.
 */
#ifndef FLCE_H_
#define FLCE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FLCE_REDUCTION_NONE = 0, /* loss is [N] per-token losses */
  FLCE_REDUCTION_SUM = 1,  /* loss is [1]: sum over tokens */
  FLCE_REDUCTION_MEAN = 2  /* loss is [1]: sum / number of non-ignored tokens (0 if none) */
} flce_reduction_t;

typedef enum {
  FLCE_OK = 0,
  FLCE_ERR_INVALID_ARG = 1,       /* a size, option or required pointer is invalid */
  FLCE_ERR_ALIGNMENT = 2,         /* a pointer or the hidden size breaks the 16-byte rules below */
  FLCE_ERR_WORKSPACE_TOO_SMALL = 3,
  FLCE_ERR_TARGET_OUT_OF_RANGE = 4, /* from flce_read_device_error */
  FLCE_ERR_CUDA = 5,              /* a CUDA runtime call failed (launch, tensor-map encode) */
  FLCE_ERR_TIMEOUT = 6,           /* from flce_read_device_error: a kernel wait gave up */
  FLCE_ERR_UNSUPPORTED = 7        /* device is not sm_103 / sizes beyond the int32 tile grid */
} flce_status_t;

/* GEMM kernel form of a call (flce_params_t.gemm_form). All forms compute
 * the same products; results differ only in the order of fp32 accumulation
 * inside a tile, not in what is summed. */
typedef enum {
  FLCE_GEMM_DEFAULT = 0,    /* library default, per GEMM: FLCE_GEMM_WIDE_PAIR where its
                               K loop has >= 4096 elements and it has >= 608 256 x 512
                               tiles, else FLCE_GEMM_CTA_PAIR (FLCE_GEMM_FORM=single|pair|
                               wide in the environment overrides the default, not an
                               explicit form) */
  FLCE_GEMM_SINGLE_CTA = 1, /* one CTA per 128 x 256 tile (tcgen05 cta_group::1) */
  FLCE_GEMM_CTA_PAIR = 2,   /* two CTAs of a cluster per 256 x 256 tile (cta_group::2) */
  FLCE_GEMM_WIDE_PAIR = 3   /* two CTAs per 256 x 512 tile (two cta_group::2 MMAs per K
                               step sharing A: a quarter fewer operand bytes per flop);
                               the dx GEMM, which has few output tiles, keeps 256 x 256 */
} flce_gemm_form_t;

/* Device error word bits (see flce_read_device_error). */
#define FLCE_DEVERR_TARGET 1
#define FLCE_DEVERR_TIMEOUT 2

typedef struct {
  int64_t N;                /* tokens (rows of x); 0 is a valid no-op */
  int64_t H;                /* hidden size; > 0 and a multiple of 8 */
  int64_t V;                /* vocabulary size; > 0 */
  int64_t ignore_index;     /* targets equal to this are ignored (any int64, default -100) */
  float label_smoothing;    /* eps in [0, 1] */
  float lse_square_scale;   /* lam >= 0 (z-loss) */
  float logit_scale;        /* s, any finite value */
  int32_t reduction;        /* flce_reduction_t */
  int32_t has_bias;         /* 1: b is given ([V] bf16) */
  int32_t dW_fp32;          /* backward: 1 = dW written as fp32, 0 = bf16 */
  int32_t db_fp32;          /* backward: 1 = db written as fp32, 0 = bf16 */
  int64_t bwd_vocab_block;  /* backward vocab block BVc (multiple of 256); 0 = library default */
  int64_t vocab_start;      /* shard calls only: first vocabulary id of W's rows */
  int64_t vocab_total;      /* shard calls only: full vocabulary size (0 = W is the whole
                               vocabulary; the plain calls require 0 or V) */
  int32_t input_fp16;       /* 0: x, W, b are bf16; 1: they are fp16 (dx, and dW / db when
                               not fp32, are then fp16 too) */
  int32_t gemm_form;        /* flce_gemm_form_t; 0 = library default */
  int64_t keep_vocab;       /* kept-block calls only: width of the kept block, the
                               vocabulary columns [0, keep_vocab) whose probabilities
                               the forward keeps (a multiple of 256; 0 = BVc; values
                               below BVc keep BVc, values >= V the whole vocabulary) */
} flce_params_t;

/* Kernel kinds reported by the traced entry points. */
typedef enum {
  FLCE_KERNEL_FWD_LSE = 0,      /* forward GEMM + online-softmax partials */
  FLCE_KERNEL_FWD_MERGE = 1,    /* partial merge -> lse, per-token loss */
  FLCE_KERNEL_FWD_FINALIZE = 2, /* ordered sum of the loss (sum / mean) */
  FLCE_KERNEL_BWD_PREP = 3,     /* per-token backward coefficients */
  FLCE_KERNEL_BWD_DLOGITS = 4,  /* recompute a vocab block's logits -> bf16 dL */
  FLCE_KERNEL_BWD_DB = 5,       /* bias-gradient partial sum of a block */
  FLCE_KERNEL_BWD_DW = 6,       /* dW block GEMM */
  FLCE_KERNEL_BWD_DX = 7,       /* dx accumulate GEMM */
  FLCE_KERNEL_BWD_CONVERT = 8   /* stored or kept probabilities -> dL (an HBM pass) */
} flce_kernel_t;

/* Optional per-kernel timing without a profiler. The caller creates
 * `capacity` CUDA events (cudaEvent_t, passed as void*) and an int32 array
 * `kinds` of the same length. A traced call records events[0] on `stream`
 * before its first launch and events[i + 1] right after launch i, whose
 * flce_kernel_t it stores in kinds[i]; `count` returns the events recorded
 * (recording stops silently at capacity). Elapsed time between events i and
 * i + 1 is launch i's time on the stream. The library keeps no reference. */
typedef struct {
  void** events;
  int32_t capacity;
  int32_t count;
  int32_t* kinds;
} flce_trace_t;

/* Workspace bytes a call needs: which = 0 for the forward calls, 1 for
 * flce_backward and flce_backward_shard, 2 for flce_backward_keep (no dL
 * block: it stages dL in the kept buffer), 3 for flce_backward_store.
 * Returns 0 for invalid parameters or N == 0. */
size_t flce_workspace_size(const flce_params_t* p, int which);

/* The GEMM form (FLCE_GEMM_SINGLE_CTA, _CTA_PAIR or _WIDE_PAIR) that calls with
 * these parameters run for one GEMM: which = 0 the forward logits GEMM, 1 the
 * backward recompute, 2 dW, 3 dx (1 and 2 for the first vocabulary block).
 * The dx GEMM runs a wide form as CTA pairs. Host only; returns -1 for NULL, invalid parameters or an invalid
 * `which`. */
int32_t flce_resolved_gemm_form(const flce_params_t* p, int32_t which);

/*
 * Forward. x: [N, H] bf16; W: [V, H] bf16; b: [V] bf16 or NULL (has_bias = 0);
 * y: [N] int64 targets in [0, V) or ignore_index.
 * Writes loss (fp32, [1] for sum/mean, [N] for none) and lse ([N] fp32,
 * natural log, for every token including ignored ones). lse is what
 * flce_backward needs from the forward pass.
 * (x, W, b are fp16 instead when input_fp16 = 1.)
 * x, W, b and the workspace must be 16-byte aligned. dev_err: one device
 * int32 (may be NULL to skip device error reporting).
 */
flce_status_t flce_forward(const flce_params_t* p, const void* x, const void* W, const void* b,
                           const int64_t* y, float* loss, float* lse, void* workspace,
                           size_t workspace_bytes, int32_t* dev_err, void* stream);

/*
 * Backward. dloss: device fp32, [1] for sum/mean or [N] for none (the
 * gradient of the caller's objective with respect to `loss`). lse: the
 * forward's [N] output. x, W, b, y as in flce_forward (the logits are
 * recomputed from them one vocabulary block at a time).
 * Writes dx [N, H] bf16, dW [V, H] (fp32 or bf16 per dW_fp32) and, when
 * has_bias, db [V] (fp32 or bf16 per db_fp32). Every element of dx, dW and db
 * is overwritten (no accumulation into the caller's buffers).
 */
flce_status_t flce_backward(const flce_params_t* p, const float* dloss, const float* lse,
                            const void* x, const void* W, const void* b, const int64_t* y,
                            void* dx, void* dW, void* db, void* workspace, size_t workspace_bytes,
                            int32_t* dev_err, void* stream);

/* flce_forward / flce_backward with an optional trace (NULL = untraced). */
flce_status_t flce_forward_traced(const flce_params_t* p, const void* x, const void* W,
                                  const void* b, const int64_t* y, float* loss, float* lse,
                                  void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                  void* stream, flce_trace_t* trace);
flce_status_t flce_backward_traced(const flce_params_t* p, const float* dloss, const float* lse,
                                   const void* x, const void* W, const void* b, const int64_t* y,
                                   void* dx, void* dW, void* db, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, void* stream,
                                   flce_trace_t* trace);

/*
 * Kept-block mode: the backward recomputes every vocabulary block but the
 * first. (Our combination of DeepSpeed PR #8792 "What", where the backward
 * recomputes the logits one vocabulary block at a time into a staged block,
 * with the grad-in-forward of Liger-Kernel commit 95b01e9, which forms the
 * gradient from logits the forward already holds.)
 *
 * flce_forward_keep computes what flce_forward does and also leaves, in the
 * caller's `kept` buffer (flce_kept_size(p) bytes, 16-byte aligned), the
 * probabilities of the first backward vocabulary block [0, BVc), where BVc is
 * the block flce_backward would use for p (bwd_vocab_block, or the library
 * default; p->keep_vocab widens the kept block, below): each 32-column
 * chunk's q = exp(z - m_c) as fp16 in an [N, BVc] array, m_c being the
 * running maximum of the row's logits up to that chunk, plus the m_c (fp32).
 * These are exponentials the forward's online softmax computes anyway.
 * flce_backward_keep turns that block into its dlogits in place (an HBM pass
 * instead of 2 N H BVc flops of recompute) and then uses the same buffer as
 * the dL staging block of the blocks it recomputes, so its workspace
 * (flce_workspace_size(p, 2)) holds no dL block: the kept buffer plus that
 * workspace take the same memory as flce_backward's workspace, plus the
 * chunk maxima. At the Llama-3 head shape (V = 128256, BVc = 65536) this
 * skips half of the recompute, an eighth of the step's flops.
 * Both calls take the same p (the kept layout depends on N, V, BVc and
 * keep_vocab); the backward consumes the kept state (it holds dL
 * afterwards), and the buffer must be left untouched between the two calls.
 * The vocabulary-shard calls have kept-block forms too (below). trace may be
 * NULL.
 */
size_t flce_kept_size(const flce_params_t* p);

/* A wider kept block (p->keep_vocab > BVc) trades memory for recompute: the
 * forward keeps the probabilities of [0, K) (K = keep_vocab, capped at the
 * vocabulary), the backward converts that block in place and then recomputes
 * the rest, [K, V), in blocks of BVc staged at the start of the kept buffer.
 * K = V is the stored mode below. flce_kept_size and
 * flce_workspace_size(p, 2) follow keep_vocab.
 *
 * flce_keep_vocab_within returns the widest keep_vocab whose kept-mode
 * memory, flce_kept_size + flce_workspace_size(., 2), stays within
 * flce_workspace_size(p, 1) + extra_bytes (the recompute backward's
 * workspace plus extra_bytes). The widths tried are the whole vocabulary,
 * then V - k BVc rounded up to 256 for k = 1, 2, ... (so the recomputed part
 * is k blocks of BVc at most), down to BVc, which is returned when nothing
 * wider fits (one block takes N BVc / 8 bytes of chunk maxima more than the
 * recompute mode). extra_bytes = 4 V H is the fp32 [V, H] dW accumulator
 * that the method's memory budget allows for and this library never
 * allocates. Host only; returns 0 for invalid parameters or N == 0. */
int64_t flce_keep_vocab_within(const flce_params_t* p, size_t extra_bytes);
flce_status_t flce_forward_keep(const flce_params_t* p, const void* x, const void* W,
                                const void* b, const int64_t* y, float* loss, float* lse,
                                void* kept, size_t kept_bytes, void* workspace,
                                size_t workspace_bytes, int32_t* dev_err, void* stream,
                                flce_trace_t* trace);
flce_status_t flce_backward_keep(const flce_params_t* p, const float* dloss, const float* lse,
                                 void* kept, size_t kept_bytes, const void* x, const void* W,
                                 const void* b, const int64_t* y, void* dx, void* dW, void* db,
                                 void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                 void* stream, flce_trace_t* trace);

/*
 * Stored-probability mode: no logits recompute in the backward pass. This is
 * the kept-block mode with one block spanning the whole vocabulary
 * (p->bwd_vocab_block and p->keep_vocab are ignored): flce_forward_store
 * keeps every logit's
 * probability, ~2 N V bytes in `saved` (flce_saved_size(p) bytes, 16-byte
 * aligned), and flce_backward_store converts it to dlogits in place and runs
 * one dW and one dx GEMM over the whole vocabulary, saving 2 N H V flops (a
 * quarter of the step) for that memory. Its workspace is
 * flce_workspace_size(p, 3). The backward consumes `saved` (it holds dL
 * afterwards); leave it untouched between the two calls. trace may be NULL.
 */
size_t flce_saved_size(const flce_params_t* p);
flce_status_t flce_forward_store(const flce_params_t* p, const void* x, const void* W,
                                 const void* b, const int64_t* y, float* loss, float* lse,
                                 void* saved, size_t saved_bytes, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream,
                                 flce_trace_t* trace);
flce_status_t flce_backward_store(const flce_params_t* p, const float* dloss, const float* lse,
                                  void* saved, size_t saved_bytes, const void* x,
                                  const void* W, const void* b, const int64_t* y, void* dx,
                                  void* dW, void* db, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_err, void* stream, flce_trace_t* trace);

/*
 * Vocabulary-parallel FLCE (DeepSpeed PR #8792, "What": each rank holds a
 * [vocab / tp] block of the LM head; forward runs one MAX and one SUM
 * all-reduce of per-token statistics, backward reduces the hidden gradient
 * in fp32 before casting). For these calls W (and b) are the rows
 * [vocab_start, vocab_start + V) of a vocab_total vocabulary (params fields),
 * shards may be uneven, and y holds global vocabulary ids on every shard.
 * The collectives themselves are the caller's (NCCL, gloo, or a host loop):
 *
 *   1. flce_forward_shard  -> stats [4, N] fp32: rows (m, d, z_y, sum_z) with
 *      m = max_v z log2(e) over the shard, d = sum_v 2^(z log2(e) - m),
 *      z_y = the target logit if y is in the shard else 0, sum_z (0 without
 *      label smoothing). Workspace: flce_workspace_size(p, 0).
 *   2. caller: M = all-reduce MAX of row 0.
 *   3. flce_shard_rescale(stats, M): d <- d 2^(m - M), m <- M.
 *   4. caller: all-reduce SUM of rows 1..3.
 *   5. flce_loss_from_stats (params with V = vocab_total and vocab_total = 0,
 *      or the shard's params) -> loss, lse exactly as flce_forward would give
 *      for the whole vocabulary. Workspace: flce_workspace_size(p, 0).
 *   6. flce_backward_shard(global lse) -> this shard's dW rows and db, and an
 *      fp32 partial dx [N, H]; caller: all-reduce SUM of dx_partial, then
 *      flce_cast_f32 (16-byte aligned src and dst) to the operand type
 *      (dst_fp16 = input_fp16) for dx.
 */
flce_status_t flce_forward_shard(const flce_params_t* p, const void* x, const void* W,
                                 const void* b, const int64_t* y, float* stats, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err, void* stream);
flce_status_t flce_shard_rescale(const flce_params_t* p, float* stats, const float* global_max,
                                 void* stream);
flce_status_t flce_loss_from_stats(const flce_params_t* p, const float* stats, const int64_t* y,
                                   float* loss, float* lse, void* workspace,
                                   size_t workspace_bytes, int32_t* dev_err, void* stream);
flce_status_t flce_backward_shard(const flce_params_t* p, const float* dloss, const float* lse,
                                  const void* x, const void* W, const void* b, const int64_t* y,
                                  float* dx_partial, void* dW, void* db, void* workspace,
                                  size_t workspace_bytes, int32_t* dev_err, void* stream);
flce_status_t flce_cast_f32(const float* src, void* dst, int64_t n, int32_t dst_fp16,
                            void* stream);

/* Steps 1 and 6 with the kept block: the shard's forward also keeps the
 * probabilities of its own first backward vocabulary block (its rows
 * [vocab_start, vocab_start + BVc), BVc per p as in flce_forward_keep), and
 * the shard's backward converts them in place instead of recomputing them.
 * kept: flce_kept_size(p) bytes for the shard's p, 16-byte aligned, consumed
 * by the backward; the backward's workspace is flce_workspace_size(p, 2). */
flce_status_t flce_forward_shard_keep(const flce_params_t* p, const void* x, const void* W,
                                      const void* b, const int64_t* y, float* stats, void* kept,
                                      size_t kept_bytes, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_err, void* stream);
flce_status_t flce_backward_shard_keep(const flce_params_t* p, const float* dloss,
                                       const float* lse, void* kept, size_t kept_bytes,
                                       const void* x, const void* W, const void* b,
                                       const int64_t* y, float* dx_partial, void* dW, void* db,
                                       void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                       void* stream);

/*
 * Forward without a workspace argument, for callers that cannot allocate
 * device memory where they compute the loss (an inference-engine plugin whose
 * enqueue step must not allocate, a service loop that forbids allocation
 * after start-up, a component beside a caching allocator that holds nearly all
 * device memory). The pages have no counterpart: this is a packaging of
 * flce_forward, not part of the method.
 *
 * Arguments and results are those of flce_forward; the scratch that
 * flce_forward takes from `workspace` comes instead from one array of
 * FLCE_NOALLOC_SCRATCH_BYTES built into the library as a static device
 * variable (every GPU that loads the library keeps it until the process
 * exits). A problem whose flce_workspace_size(p, 0) exceeds that size is
 * rejected with FLCE_ERR_WORKSPACE_TOO_SMALL before anything runs.
 * The first call on each device looks up the array's device address with
 * that device current; make that first call before any stream capture.
 * The address is kept for the life of the process, so do not use this entry
 * point across a cudaDeviceReset of that device (the reset unloads the
 * library's module and the kept address would no longer be the array's).
 * The call allocates and frees nothing. All calls share the one array, so
 * calls that overlap on the GPU (e.g. on two streams) race on it: order them.
 * Each call writes every scratch value it later reads, so stale contents from
 * an earlier call never leak into a result.
 */
#define FLCE_NOALLOC_SCRATCH_BYTES (64 * 1024 * 1024)
flce_status_t flce_forward_noalloc(const flce_params_t* p, const void* x, const void* W,
                                   const void* b, const int64_t* y, float* loss, float* lse,
                                   int32_t* dev_err, void* stream);

/* Failure-detection self-test: launches one kernel that waits, through the
 * same bounded mbarrier wait the GEMM pipelines use, on a barrier nothing
 * arrives on. After limit_cycles (1 .. 2^32 SM clock cycles) the wait gives
 * up and ORs FLCE_DEVERR_TIMEOUT into *dev_err; the kernel returns normally,
 * so flce_read_device_error then reports FLCE_ERR_TIMEOUT and the CUDA
 * context stays usable. (The pipelines' own limit is about one second.) */
flce_status_t flce_selftest_wait_timeout(int32_t* dev_err, int64_t limit_cycles, void* stream);

/* Synchronises `stream`, reads the device error word into *host_err (HOST
 * pointer, may be NULL), clears the device word and maps it to a status:
 * FLCE_OK, FLCE_ERR_TARGET_OUT_OF_RANGE or FLCE_ERR_TIMEOUT. */
flce_status_t flce_read_device_error(int32_t* dev_err, void* stream, int32_t* host_err);

/* Static string for a status code. */
const char* flce_status_string(flce_status_t status);

/* Library version, e.g. "0.1.0". */
const char* flce_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FLCE_H_ */
