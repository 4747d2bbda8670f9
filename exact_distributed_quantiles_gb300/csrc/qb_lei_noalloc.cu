// qb_lei_noalloc.cu -- lei_inject_noalloc: load-error injection for callers
// that cannot provide a scratch workspace.
//
// lei_inject needs a small device workspace (eta * rho per local batch and
// expert) that the caller allocates.  Some callers cannot allocate device
// memory at the call site: code running under a framework whose caching
// allocator owns the whole memory pool (a stray cudaMalloc would bypass it or
// fail), services that fix their device-memory budget at start-up, or
// callers that simply hold no allocator handle where LEI is applied.  This
// entry point keeps that scratch in a fixed-size array in the library's own
// device memory instead and allocates nothing.
//
// The array is a file-scope __device__ variable.  Its name is only a host-side
// stand-in in host code, so the device address is looked up with
// cudaGetSymbolAddress, with the device current, on the first successful call
// made on that device.  Under CUDA's lazy module loading (the default) that
// lookup is also what loads this library's device code on the device and
// reserves the array (kScratchFloats * 4 bytes); under eager loading
// (CUDA_MODULE_LOADING=EAGER) the reservation happens when the library's
// context is set up.  Either way the array then stays until the process exits.
#include <mutex>

#include "qb_internal.h"

namespace qb {
namespace {

constexpr int64_t kScratchFloats = 65536;  // num_batches * E must not exceed this

static __device__ __align__(256) float g_lei_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float* g_scratch[kMaxDevices] = {};

// Device address of g_lei_scratch on the current device, or nullptr.  Only a
// successful lookup is cached: after a failure (for instance a first call made
// inside a stream capture) the error is cleared and the next call tries again.
float* scratch_on_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_lei_scratch) == cudaSuccess) {
      g_scratch[dev] = static_cast<float*>(p);
    } else {
      (void)cudaGetLastError();
    }
  }
  return g_scratch[dev];
}

}  // namespace
}  // namespace qb

extern "C" int lei_inject_noalloc(float* grad, const int32_t* topk_idx, int64_t N, int E, int k,
                                  float eta, int64_t batch_tokens, void* stream) {
  using namespace qb;
  if (!grad || !topk_idx) return QB_EINVAL;
  if (!aligned16(grad)) return QB_EINVAL;
  if (N < 0 || batch_tokens < 0) return QB_EINVAL;
  if (!supported_E(E)) return QB_EUNSUPPORTED;
  if (k < 1 || k >= E) return QB_EINVAL;
  if (N == 0) return QB_OK;
  if (batch_tokens == 0 || batch_tokens > N) batch_tokens = N;
  if (N > INT32_MAX) return QB_EOVERFLOW;
  const int64_t nb = (N + batch_tokens - 1) / batch_tokens;
  if (nb > kScratchFloats / E) return QB_EINVAL;  // scratch would not hold num_batches * E
  float* scratch = scratch_on_current_device();
  if (!scratch) return QB_ECUDA;
  // Every batch row of the scratch is written in full by the first kernel
  // before the second reads it, so nothing needs clearing between calls.
  return launch_lei(grad, topk_idx, N, E, k, eta, batch_tokens, scratch, as_stream(stream));
}
