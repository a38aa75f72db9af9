// Tensor-core (tcgen05 / TMEM / TMA) kernels for bf16, dk = dv = 128, chunk 64.
// Until they are in place every shape takes the CUDA-core kernels.

#include "gdn.h"
#include "gdn_internal.cuh"

namespace gdn {

// Per-device status word: bounded device-side waits record a timeout here.
__device__ int g_device_status = 0;

cudaError_t read_and_clear_device_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  if (e != cudaSuccess) return e;
  *status = v;
  return cudaSuccess;
}

bool tc_supported(const Problem&) { return false; }
size_t tc_bwd_workspace(const Problem&) { return 0; }
cudaError_t tc_fwd(const Problem&, cudaStream_t) { return cudaErrorNotSupported; }
cudaError_t tc_bwd(const Problem&, cudaStream_t) { return cudaErrorNotSupported; }

}  // namespace gdn
