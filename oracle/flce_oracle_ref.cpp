// CPU fp64 reference of fused linear cross-entropy (FLCE), in plain C++.
//
// TEST INFRASTRUCTURE. Only the tests load this library (through
// oracle/cpp.py); the GPU library never does and shares no code with it. It
// is a second, independent statement of the same definition as
// oracle/flce_oracle.py, written as loops over the bf16- (or fp16-) rounded
// inputs widened exactly to double, with every product and sum in double.
// It holds the whole [N, V] matrix of logit gradients, so it is meant for the
// small problems the tests give it.
//
// What it computes, per token row n (the plain definition):
//   z[n, v]  = s * (sum_h x[n, h] W[v, h] + b[v])
//   lse[n]   = M + log sum_v exp(z[n, v] - M),  M = max_v z[n, v]
//   l[n]     = (1 - eps)(lse[n] - z[n, y_n]) + eps lse[n]
//              - (eps / V) sum_v z[n, v] + lam lse[n]^2        (0 if y_n ignored)
//   loss     = l (none) | sum_n l[n] (sum) | sum_n l[n] / total (mean; 0 if total = 0)
//   g[n]     = dloss[n] (none) | dloss (sum) | dloss / total (mean); 0 if ignored
//   dz[n, v] = g[n] ((1 + 2 lam lse[n]) exp(z[n, v] - lse[n]) - eps / V
//                    - (1 - eps) [v == y_n])
//   dx = s dz W,  dW = s dz^T x,  db = s sum_n dz[n, :]
//
// Sources, by page and section:
//   * flash-linear-attention, fla/modules/fused_linear_cross_entropy.py:
//     fused_linear_cross_entropy_forward (logits from F.linear, then the
//     logit_scale; total = the non-ignored count) and cross_entropy_kernel
//     (ignored rows get zero loss and gradient; loss = lse - z_y; label
//     smoothing with eps / V; mean divides by total).
//   * Liger-Kernel PR #239 "Support Z Loss in CE", "Details": the per-token
//     z-loss lam lse^2 and the derivative (1 + 2 lam lse) softmax - eps / K
//     - (1 - eps) delta.
//   * DeepSpeed PR #8792 "What": reduction "none" beside sum and mean.
//
// Parity: pinned by tests/test_oracle_cpp.py against the hand-derived closed
// forms of tests/golden/closed_form_cases.json, the numpy oracle on random
// problems with every option, and the invariant sum_v dz[n, v] = 2 lam g[n]
// lse[n].
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <thread>
#include <vector>

namespace {

enum { kNone = 0, kSum = 1, kMean = 2 };

struct Problem {
  int64_t N, H, V;
  const double *x, *W, *b;
  const int64_t* y;
  int64_t ignore_index;
  double eps, lam, s;
};

// Runs f(i) for i in [0, n) on `threads` threads (contiguous ranges).
template <class F>
void parallel_for(int64_t n, int threads, F f) {
  if (threads < 2 || n < 2) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  const int t = static_cast<int>(std::min<int64_t>(threads, n));
  std::vector<std::thread> pool;
  for (int k = 0; k < t; ++k)
    pool.emplace_back([=] {
      for (int64_t i = n * k / t; i < n * (k + 1) / t; ++i) f(i);
    });
  for (auto& th : pool) th.join();
}

// Logits of one token row.
void logits_row(const Problem& p, int64_t n, double* z) {
  for (int64_t v = 0; v < p.V; ++v) {
    double acc = 0.0;
    for (int64_t h = 0; h < p.H; ++h) acc += p.x[n * p.H + h] * p.W[v * p.H + h];
    if (p.b) acc += p.b[v];
    z[v] = p.s * acc;
  }
}

double logsumexp(const double* z, int64_t V) {
  double m = z[0];
  for (int64_t v = 1; v < V; ++v) m = std::max(m, z[v]);
  double d = 0.0;
  for (int64_t v = 0; v < V; ++v) d += std::exp(z[v] - m);
  return m + std::log(d);
}

bool ignored(const Problem& p, int64_t n) { return p.y[n] == p.ignore_index; }

int64_t total(const Problem& p) {
  int64_t t = 0;
  for (int64_t n = 0; n < p.N; ++n) t += ignored(p, n) ? 0 : 1;
  return t;
}

bool valid(const Problem& p, int reduction) {
  if (p.N < 0 || p.H <= 0 || p.V <= 0 || !p.W || !p.y || (p.N > 0 && !p.x)) return false;
  if (reduction < kNone || reduction > kMean) return false;
  for (int64_t n = 0; n < p.N; ++n)
    if (!ignored(p, n) && (p.y[n] < 0 || p.y[n] >= p.V)) return false;
  return true;
}

}  // namespace

extern "C" {

// loss: [N] (none) or [1]; lse: [N]. Returns 0, or 1 for invalid arguments
// (including a target outside [0, V) that is not ignore_index).
int flce_ref_forward(int64_t N, int64_t H, int64_t V, const double* x, const double* W,
                     const double* b, const int64_t* y, int64_t ignore_index, double eps,
                     double lam, double s, int reduction, int threads, double* loss,
                     double* lse) {
  const Problem p{N, H, V, x, W, b, y, ignore_index, eps, lam, s};
  if (!valid(p, reduction) || !loss || (N > 0 && !lse)) return 1;
  std::vector<double> token(static_cast<size_t>(N), 0.0);
  parallel_for(N, threads, [&](int64_t n) {
    std::vector<double> z(static_cast<size_t>(V));
    logits_row(p, n, z.data());
    lse[n] = logsumexp(z.data(), V);
    if (ignored(p, n)) return;
    double sum_z = 0.0;
    for (int64_t v = 0; v < V; ++v) sum_z += z[v];
    const double l = lse[n];
    token[n] = (1.0 - eps) * (l - z[y[n]]) + eps * l - (eps / V) * sum_z + lam * l * l;
  });
  if (reduction == kNone) {
    for (int64_t n = 0; n < N; ++n) loss[n] = token[n];
    return 0;
  }
  double acc = 0.0;  // in row order
  for (int64_t n = 0; n < N; ++n) acc += token[n];
  const int64_t t = total(p);
  loss[0] = reduction == kSum ? acc : (t > 0 ? acc / t : 0.0);
  return 0;
}

// dloss: [N] (none) or [1]. dx [N, H], dW [V, H], db [V] (may be null when
// b is null). Returns 0, or 1 for invalid arguments.
int flce_ref_backward(int64_t N, int64_t H, int64_t V, const double* x, const double* W,
                      const double* b, const int64_t* y, int64_t ignore_index, double eps,
                      double lam, double s, int reduction, const double* dloss, int threads,
                      double* dx, double* dW, double* db) {
  const Problem p{N, H, V, x, W, b, y, ignore_index, eps, lam, s};
  if (!valid(p, reduction) || !dloss || !dW || (N > 0 && !dx) || (b && !db)) return 1;
  const int64_t t = total(p);
  // dz [N, V], row by row.
  std::vector<double> dz(static_cast<size_t>(N) * V, 0.0);
  parallel_for(N, threads, [&](int64_t n) {
    if (ignored(p, n)) return;
    double g = reduction == kNone ? dloss[n] : dloss[0];
    if (reduction == kMean) g = t > 0 ? g / t : 0.0;
    std::vector<double> z(static_cast<size_t>(V));
    logits_row(p, n, z.data());
    const double l = logsumexp(z.data(), V);
    double* row = dz.data() + n * V;
    for (int64_t v = 0; v < V; ++v) {
      const double target = v == y[n] ? 1.0 : 0.0;
      row[v] = g * ((1.0 + 2.0 * lam * l) * std::exp(z[v] - l) - eps / V - (1.0 - eps) * target);
    }
  });
  // dx = s dz W (row n of dx sums over the vocabulary).
  parallel_for(N, threads, [&](int64_t n) {
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t v = 0; v < V; ++v) acc += dz[n * V + v] * W[v * H + h];
      dx[n * H + h] = s * acc;
    }
  });
  // dW = s dz^T x and db = s sum_n dz (row v sums over the tokens).
  parallel_for(V, threads, [&](int64_t v) {
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += dz[n * V + v] * x[n * H + h];
      dW[v * H + h] = s * acc;
    }
    if (db) {
      double acc = 0.0;
      for (int64_t n = 0; n < N; ++n) acc += dz[n * V + v];
      db[v] = s * acc;
    }
  });
  return 0;
}

}  // extern "C"
