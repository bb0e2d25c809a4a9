// forge_no_alloc.cu -- forge_backward_step_no_alloc: the fused backward
// pass (input gradient + weight-gradient step, one read of W) for callers
// that cannot allocate device memory. The fused path needs scratch for its
// per-column dX partial sums; here that scratch is a fixed array compiled
// into the library instead of a buffer the caller passes in.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/forge.h"

namespace forge {
forge_status set_error(forge_status st, const char* msg);
}

namespace {

// 64 MiB: enough for every Llama-3.1-8B projection at BT <= 512 on a
// 152-SM GPU (the down-projection, the largest, needs 57 MiB). Each GPU
// that loads this part of the library keeps the array until the process
// exits.
constexpr size_t kScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char forge_no_alloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is asked of the
// runtime, once per device, with that device current. Under lazy module
// loading this first lookup is when the driver loads the module on the device
// and reserves the array, so it is the call that can run out of memory. The
// cached address belongs to the device's current context: a cudaDeviceReset
// leaves it stale (the header tells callers not to reset and call again).
forge_status scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return forge::set_error(FORGE_ERR_CUDA, "backward_step_no_alloc: cudaGetDevice failed");
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, forge_no_alloc_scratch);
    if (e != cudaSuccess) {
      char msg[256];
      snprintf(msg, sizeof(msg), "backward_step_no_alloc: cudaGetSymbolAddress of the scratch array: %s",
               cudaGetErrorString(e));
      return forge::set_error(FORGE_ERR_CUDA, msg);
    }
    g_scratch[dev] = p;
  }
  *out = g_scratch[dev];
  return FORGE_OK;
}

}  // namespace

extern "C" forge_status forge_backward_step_no_alloc(forge_rule rule, const forge_tensor* X, const forge_tensor* dY,
                                                     forge_tensor* W, forge_tensor* s0, forge_tensor* s1,
                                                     forge_tensor* dX, const forge_hyper* h, int64_t step,
                                                     uint64_t seed, forge_stream_t stream) {
  if (X == nullptr || dY == nullptr || h == nullptr)
    return forge::set_error(FORGE_ERR_INVALID_ARG, "backward_step_no_alloc: null argument");
  const size_t need = forge_workspace_bytes(dY->cols, X->cols, X->rows);
  if (need > kScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "backward_step_no_alloc: this layer needs %zu bytes of scratch; the built-in array holds %zu "
             "(use forge_backward_step with a workspace of forge_workspace_bytes() bytes)",
             need, kScratchBytes);
    return forge::set_error(FORGE_ERR_UNSUPPORTED, msg);
  }
  void* ws = nullptr;
  const forge_status st = scratch_address(&ws);
  if (st != FORGE_OK) return st;
  // The fused path only: the split path needs no scratch and is
  // forge_backward_step's to choose.
  forge_hyper hf = *h;
  hf.flags = (hf.flags & ~FORGE_FLAG_BACKWARD_SPLIT) | FORGE_FLAG_BACKWARD_FUSED;
  return forge_backward_step(rule, X, dY, W, s0, s1, dX, &hf, step, seed, ws, kScratchBytes, stream);
}
