// flce_forward_noalloc: the forward pass with its scratch memory taken from
// a fixed array inside this library instead of a caller-supplied workspace.
//
// Who needs it: code that must not allocate device memory at the point where
// it computes the loss, for example an inference-engine plugin whose enqueue
// step is not allowed to allocate, a hot loop in a service that forbids
// allocation after start-up, or a component running next to a caching
// allocator that already holds almost all device memory, where a fresh
// cudaMalloc can fail or fragment the pool. Such callers still own the
// inputs and outputs; this entry point only removes the workspace.
//
// The scratch is one static __device__ array of FLCE_NOALLOC_SCRATCH_BYTES
// (64 MiB). Every GPU that loads this library holds it until the process
// exits. All calls share it, so calls whose kernels overlap on the GPU (for
// example on two streams) race on it and must be ordered by the caller.
// Every scratch value a call reads is first written by that same call, so
// nothing is cleared between calls.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/flce.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[FLCE_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// The name g_scratch is only a host-side handle; the device address comes
// from cudaGetSymbolAddress, looked up once per device with that device
// current (the first call on each device does it). The address is kept for
// the life of the process: a cudaDeviceReset would invalidate it, and the
// header tells callers not to use this entry point across one.
flce_status_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FLCE_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FLCE_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return FLCE_ERR_CUDA;
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return FLCE_OK;
}

}  // namespace

extern "C" flce_status_t flce_forward_noalloc(const flce_params_t* p, const void* x,
                                              const void* W, const void* b, const int64_t* y,
                                              float* loss, float* lse, int32_t* dev_err,
                                              void* stream) {
  if (!p) return FLCE_ERR_INVALID_ARG;
  const size_t need = flce_workspace_size(p, 0);
  if (need > static_cast<size_t>(FLCE_NOALLOC_SCRATCH_BYTES)) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  if (need == 0)  // N == 0 or invalid parameters: nothing needs scratch
    return flce_forward(p, x, W, b, y, loss, lse, nullptr, 0, dev_err, stream);
  void* scratch = nullptr;
  const flce_status_t st = scratch_for_current_device(&scratch);
  if (st != FLCE_OK) return st;
  return flce_forward(p, x, W, b, y, loss, lse, scratch, FLCE_NOALLOC_SCRATCH_BYTES, dev_err,
                      stream);
}
