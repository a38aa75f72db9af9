// Internal declarations shared by the C-ABI layer and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

namespace gdn {

// Everything one launch of the mixer needs.  Token tensors are [B,T,H,D],
// states [B,H,dk,dv]; see include/gdn.h.
struct Problem {
  int B, T, H, dk, dv, C, N;  // N = ceil(T / C) chunks per sequence
  bool kda, bf16;
  bool no_delta;  // the Mamba2 mixer: the state only accumulates beta k v^T (no delta rule)
  const void *q, *k, *v, *do_;
  const float *g, *beta, *h0, *dht;
  void *o, *dq, *dk_, *dv_;
  float *ht, *dg, *dbeta, *dh0;
  void* ws;
  size_t ws_bytes;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// CUDA-core fp32 kernels (any dk, dv <= 128; chunk 16/32/64).
size_t simt_bwd_workspace(const Problem& p);
// save / saved: the workspace is a saved context (simt_bwd_workspace bytes);
// the forward writes every chunk's fp32 entry state into it and the backward
// reads them instead of running the states pass.
// only: if non-NULL, a per-sequence flag array [B*H]; the kernels then run
// only the sequences whose flag is set (the others' outputs are untouched).
cudaError_t simt_fwd(const Problem& p, cudaStream_t s, bool save, const int* only = nullptr);
cudaError_t simt_bwd(const Problem& p, cudaStream_t s, bool saved, const int* only = nullptr);

// Tensor-core kernels (bf16, dk = dv = 128, chunk = 64).
bool tc_supported(const Problem& p);
size_t tc_fwd_workspace(const Problem& p);
size_t tc_bwd_workspace(const Problem& p);
size_t tc_ctx_bytes(const Problem& p);
// save / saved: the workspace is a saved context (tc_ctx_bytes) that the
// forward fills and the backward of the same inputs reads.
cudaError_t tc_fwd(const Problem& p, cudaStream_t s, bool save);
cudaError_t tc_bwd(const Problem& p, cudaStream_t s, bool saved);

// KDA tensor-core kernels (bf16, dk = dv = 128, chunk = 64).  Sequences
// with a chunk whose per-dimension gate range is too wide for them are
// flagged and computed by the CUDA-core kernels inside the same calls.
bool kda_tc_supported(const Problem& p);
size_t kda_tc_fwd_workspace(const Problem& p);
size_t kda_tc_bwd_workspace(const Problem& p);  // also the saved context
cudaError_t kda_tc_fwd(const Problem& p, cudaStream_t s, bool save);
cudaError_t kda_tc_bwd(const Problem& p, cudaStream_t s, bool saved);
cudaError_t kda_read_and_clear_status(int* status);

// Token-recurrent forward for a few tokens per sequence (any dk, dv <= 128).
cudaError_t decode(const Problem& p, cudaStream_t s);

// Kernel ids reported by the timing hook (gdn_profile_*).
enum KernelId {
  kSimtFwd = 0,
  kSimtStates = 1,
  kSimtBwd = 2,
  kSimtBwdReduce = 3,
  kTcFwd = 4,
  kTcStates = 5,
  kTcBwd = 6,
  kTcSolve = 7,
  kTcSegment = 8,
  kTcCombine = 9,
  kDecode = 10,
  kKdaPrep = 11,
  kKdaFwd = 12,
  kKdaStates = 13,
  kKdaBwd = 14,
  kNumKernelIds = 15
};
const char* kernel_name(int id);

// Called around every kernel launch of the library (no-ops unless the calling
// thread enabled the timing hook).
void prof_before(cudaStream_t s);
void prof_after(cudaStream_t s, int kernel_id);

// Per-device status word written by bounded device-side waits.
cudaError_t read_and_clear_device_status(int* status);

// One CTA whose bounded wait runs out on purpose (see gdn_wait_selftest).
cudaError_t wait_selftest(int max_tries, cudaStream_t s);

// Records e as the calling thread's last CUDA error (what gdn_last_cuda_error
// returns) and returns GDN_ERR_CUDA.
int record_cuda_error(cudaError_t e);

}  // namespace gdn
