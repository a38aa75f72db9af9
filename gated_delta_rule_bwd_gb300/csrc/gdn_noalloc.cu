// gdn_bwd_noalloc: the GDN backward pass for callers that cannot allocate
// device memory.
//
// Who needs it: code that runs where cudaMalloc is not available or not
// allowed -- an allocator hook or memory-pool callback that must not recurse
// into the allocator, a host thread running inside a framework that owns all
// device memory and hands out only tensors, or a real-time path that forbids
// allocation after start-up.  gdn_bwd wants a caller-provided workspace
// (chunk-boundary states and partial sums); such callers have nowhere to get
// it from.  This entry point supplies that workspace from a fixed array that
// lives in the library's device image instead.
//
// The scratch array is kScratchBytes (32 MiB) of device memory that every GPU
// which loads this library keeps until the process exits.  Shapes whose
// gdn_bwd_workspace() exceeds it are refused with GDN_ERR_WORKSPACE before
// anything is launched.  All calls share the one array: two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on it and give wrong results.  The array keeps whatever the
// last call left in it; the kernels write every scratch word before reading
// it, so nothing needs clearing between calls.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress (which can load the module on that device) and
// keeps it for the life of the process.  Make that first call before
// capturing any stream into a CUDA graph.  A cudaDeviceReset after it would
// leave the kept address stale, so it is not supported.

#include <mutex>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace {

constexpr size_t kScratchBytes = 32u << 20;
constexpr int kMaxDevices = 64;

// File-scope device scratch.  Host code must not pass `g_noalloc_scratch`
// itself to a kernel: on the host that name is only a stand-in, not a device
// address.  The address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up once per
// device).  Returns cudaSuccess and fills *out, or the CUDA error.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" GDN_API int gdn_bwd_noalloc(const gdn_shape* shape, const void* q, const void* k,
                               const void* v, const float* g, const float* beta,
                               const float* h0, const void* do_, const float* dht, void* dq,
                               void* dk, void* dv, float* dg, float* dbeta, float* dh0,
                               void* stream) {
  if (!shape) return GDN_ERR_ARG;
  const size_t need = gdn_bwd_workspace(shape);
  if (need > kScratchBytes) return GDN_ERR_WORKSPACE;
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return gdn::record_cuda_error(e);  // set-up failed
  return gdn_bwd(shape, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, scratch,
                 kScratchBytes, stream);
}
