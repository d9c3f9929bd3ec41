/* A C program driving the FLCE C ABI directly (no Python): the caller
 * allocates every buffer, the library allocates nothing.
 *
 * Closed form used as the check: with W = 0 and no bias every logit is 0, so
 * lse = log V, the mean loss is log V, dx = 0 and, for reduction mean over T
 * non-ignored tokens, dW[v, :] = s * sum_n (1/V - [v == y_n]) x[n, :] / T
 * (gradient of cross-entropy at uniform logits; fla cross_entropy_kernel).
 * Run three times: the plain forward / backward, the kept-block pair, and
 * the kept-block pair with a kept block of 512 columns (keep_vocab). */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "flce.h"

static uint16_t f2bf(float f) { uint32_t u; memcpy(&u, &f, 4); return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16); }
static float bf2f(uint16_t b) { uint32_t u = (uint32_t)b << 16; float f; memcpy(&f, &u, 4); return f; }

#define CK(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { fprintf(stderr, "cuda %s at %d\n", cudaGetErrorString(e_), __LINE__); return 2; } } while (0)
#define FL(x) do { flce_status_t s_ = (x); if (s_ != FLCE_OK) { fprintf(stderr, "flce %s at %d\n", flce_status_string(s_), __LINE__); return 3; } } while (0)

/* One forward + backward (plain, or the kept-block pair with 256-column
 * vocabulary blocks; keep = 2 keeps [0, 512) and recomputes the rest)
 * checked against the closed form. */
static int run(int keep) {
  const int64_t N = 200, H = 72, V = 1000;
  flce_params_t p;
  memset(&p, 0, sizeof(p));
  p.N = N; p.H = H; p.V = V; p.ignore_index = -100; p.logit_scale = 0.5f;
  p.reduction = FLCE_REDUCTION_MEAN; p.dW_fp32 = 1; p.db_fp32 = 1;
  if (keep) p.bwd_vocab_block = 256;
  if (keep == 2) {
    p.keep_vocab = 512;
    /* the budget rule answers with a width the keep calls accept */
    const int64_t kw = flce_keep_vocab_within(&p, (size_t)(4 * V * H));
    if (kw < 256 || kw % 256 != 0) { fprintf(stderr, "keep_vocab_within %lld\n", (long long)kw); return 4; }
  }

  uint16_t* hx = malloc(N * H * 2);
  int64_t* hy = malloc(N * 8);
  int64_t T = 0;
  for (int64_t i = 0; i < N * H; ++i) hx[i] = f2bf((float)((i * 37) % 17) / 8.0f - 1.0f);
  for (int64_t n = 0; n < N; ++n) { hy[n] = (n % 7 == 3) ? -100 : (n * 131) % V; T += hy[n] != -100; }

  void *x, *W, *ws_f, *ws_b, *dx, *kept = NULL; int64_t* y; float *loss, *lse, *dloss, *dW; int32_t* err;
  size_t wf = flce_workspace_size(&p, 0), wb = flce_workspace_size(&p, keep ? 2 : 1);
  size_t wk = keep ? flce_kept_size(&p) : 0;
  CK(cudaMalloc(&x, N * H * 2)); CK(cudaMalloc(&W, V * H * 2)); CK(cudaMalloc((void**)&y, N * 8));
  CK(cudaMalloc((void**)&loss, 4)); CK(cudaMalloc((void**)&lse, N * 4)); CK(cudaMalloc((void**)&dloss, 4));
  CK(cudaMalloc(&dx, N * H * 2)); CK(cudaMalloc((void**)&dW, V * H * 4)); CK(cudaMalloc((void**)&err, 4));
  CK(cudaMalloc(&ws_f, wf)); CK(cudaMalloc(&ws_b, wb));
  if (keep) CK(cudaMalloc(&kept, wk));
  CK(cudaMemcpy(x, hx, N * H * 2, cudaMemcpyHostToDevice));
  CK(cudaMemset(W, 0, V * H * 2));
  CK(cudaMemcpy(y, hy, N * 8, cudaMemcpyHostToDevice));
  float one = 1.0f;
  CK(cudaMemcpy(dloss, &one, 4, cudaMemcpyHostToDevice));
  CK(cudaMemset(err, 0, 4));

  if (keep) {
    FL(flce_forward_keep(&p, x, W, NULL, y, loss, lse, kept, wk, ws_f, wf, err, NULL, NULL));
    FL(flce_backward_keep(&p, dloss, lse, kept, wk, x, W, NULL, y, dx, dW, NULL, ws_b, wb, err,
                          NULL, NULL));
  } else {
    FL(flce_forward(&p, x, W, NULL, y, loss, lse, ws_f, wf, err, NULL));
    FL(flce_backward(&p, dloss, lse, x, W, NULL, y, dx, dW, NULL, ws_b, wb, err, NULL));
  }
  int32_t herr = 0;
  FL(flce_read_device_error(err, NULL, &herr));

  float hloss; float* hlse = malloc(N * 4); uint16_t* hdx = malloc(N * H * 2); float* hdW = malloc(V * H * 4);
  CK(cudaMemcpy(&hloss, loss, 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hlse, lse, N * 4, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdx, dx, N * H * 2, cudaMemcpyDeviceToHost));
  CK(cudaMemcpy(hdW, dW, V * H * 4, cudaMemcpyDeviceToHost));

  const double logV = log((double)V);
  int bad = 0;
  if (fabs(hloss - logV) > 1e-3 * logV) { fprintf(stderr, "loss %f != log V %f\n", hloss, logV); bad = 1; }
  for (int64_t n = 0; n < N; ++n)
    if (fabs(hlse[n] - logV) > 1e-3 * logV) { fprintf(stderr, "lse[%lld] %f\n", (long long)n, hlse[n]); bad = 1; break; }
  for (int64_t i = 0; i < N * H; ++i)
    if (bf2f(hdx[i]) != 0.0f) { fprintf(stderr, "dx[%lld] != 0\n", (long long)i); bad = 1; break; }
  double num = 0, den = 0, mx = 0, mref = 0;
  for (int64_t v = 0; v < V; ++v)
    for (int64_t h = 0; h < H; ++h) {
      double ref = 0;
      for (int64_t n = 0; n < N; ++n) {
        if (hy[n] == -100) continue;
        ref += (1.0 / V - (hy[n] == v ? 1.0 : 0.0)) * bf2f(hx[n * H + h]);
      }
      ref *= 0.5 / (double)T;
      double d = hdW[v * H + h] - ref;
      num += d * d; den += ref * ref;
      if (fabs(d) > mx) mx = fabs(d);
      if (fabs(ref) > mref) mref = fabs(ref);
    }
  if (sqrt(num / den) > 5e-3 || mx > mref / 128.0) { fprintf(stderr, "dW rel-Frobenius %g max %g\n", sqrt(num / den), mx); bad = 1; }
  if (herr != 0) { fprintf(stderr, "device error %d\n", herr); bad = 1; }
  printf("%s (%s): loss %.6f (log V %.6f), %s\n", bad ? "FAIL" : "ok",
         keep == 2 ? "kept block of 512 columns" : keep ? "kept block" : "plain", hloss, logV,
         flce_version());
  cudaFree(x); cudaFree(W); cudaFree(y); cudaFree(loss); cudaFree(lse); cudaFree(dloss);
  cudaFree(dx); cudaFree(dW); cudaFree(err); cudaFree(ws_f); cudaFree(ws_b);
  if (kept) cudaFree(kept);
  free(hx); free(hy); free(hlse); free(hdx); free(hdW);
  return bad;
}

int main(void) {
  int bad = run(0);
  bad |= run(1);
  bad |= run(2);
  return bad;
}
