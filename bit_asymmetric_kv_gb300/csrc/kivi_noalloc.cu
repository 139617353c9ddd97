// kivi_noalloc.cu -- kivi_decode_attention for callers that cannot allocate device
// memory.
//
// Some callers cannot call cudaMalloc at decode time: an allocator that must not be
// re-entered from inside a serving loop, a host process whose device memory is
// fully reserved up front, or code running where a stray allocation would break a
// memory budget.  This entry point takes its decode workspace from a fixed array
// compiled into the library instead of from the caller.
//
// The array lives in device global memory for the whole life of the process, on
// every GPU that loads the library.  Its address is looked up with
// cudaGetSymbolAddress (the array's name in host code is only a host-side handle,
// not a device address), once per device, the first time the entry point runs on
// that device.  That first call therefore performs a runtime query and should be
// made before any stream capture.  The looked-up address is kept for the life of
// the process: after a cudaDeviceReset of a device the entry point must not be used
// on that device again.  Every call shares the array: calls whose kernels overlap
// on the GPU (different streams, or different threads on the same device) race on
// it.  The decode kernels fully overwrite the part of the array they read, so
// nothing needs clearing between calls.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kivi.h"
#include "kivi_internal.h"

namespace {

// Largest workspace served from the built-in array: 8 MiB.
constexpr size_t kNoAllocBytes = size_t(8) << 20;
static __device__ __align__(256) float g_noalloc_ws[kNoAllocBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_lock;
void *g_addr[kMaxDevices] = {};

// Device address of g_noalloc_ws on the current device (looked up once per device).
cudaError_t noalloc_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> guard(g_lock);
  if (!g_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_ws);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t kivi_decode_attention_noalloc_max_workspace(void) { return kNoAllocBytes; }

int kivi_decode_attention_noalloc(const kivi_dims *d, const kivi_cache *c, const uint16_t *q, int32_t Hq,
                                  float softmax_scale, uint16_t *out, cudaStream_t st) {
  // Every argument check of the workspace entry point, in its order, without a
  // launch: given no workspace it returns KIVI_ERR_WORKSPACE exactly when all the
  // other arguments are valid, and the first failing check's status otherwise.
  const int s = kivi_decode_attention(d, c, q, Hq, softmax_scale, out, nullptr, 0, st);
  if (s != KIVI_ERR_WORKSPACE) return s;
  const size_t need = kivi_decode_workspace_bytes(d, Hq, c->n_tokens);
  if (need == 0) return KIVI_ERR_CUDA;  // the sizes passed the checks: only a device query can fail here
  if (need > kNoAllocBytes) return KIVI_ERR_WORKSPACE;
  void *ws = nullptr;
  if (noalloc_address(&ws) != cudaSuccess) return KIVI_ERR_CUDA;
  return kivi_decode_attention(d, c, q, Hq, softmax_scale, out, ws, kNoAllocBytes, st);
}

}  // extern "C"
