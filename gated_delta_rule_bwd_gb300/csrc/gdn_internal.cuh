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
  bool g16;       // KDA gate g and dg in bf16 (carried in the float pointers below)
  bool no_delta;  // the Mamba2 mixer: the state only accumulates beta k v^T (no delta rule)
  const void *q, *k, *v, *do_;
  const float *g, *beta, *h0, *dht;
  void *o, *dq, *dk_, *dv_;
  float *ht, *dg, *dbeta, *dh0;
  void* ws;
  size_t ws_bytes;
  // Packed variable-length sequences (B = 1, T = all tokens): sequence s is
  // tokens [cu_seqlens[s], cu_seqlens[s+1]); nullptr for a batch of B rows of
  // T tokens.  chunk_off (device, in the workspace) holds the first global
  // chunk of each sequence, written by the set-up kernel.
  const int* cu_seqlens;
  int nseq;
  const int* chunk_off;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Element i of the gate g (fp32, or bf16 when g16) and a store into dg.
__device__ __forceinline__ float gate_load(const Problem& p, size_t i) {
  return p.g16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(p.g)[i]) : p.g[i];
}
__device__ __forceinline__ void dgate_store(const Problem& p, size_t i, float v) {
  if (p.g16)
    reinterpret_cast<__nv_bfloat16*>(p.dg)[i] = __float2bfloat16_rn(v);
  else
    p.dg[i] = v;
}

// Number of sequences (batch rows, or packed sequences).
inline int num_seqs(const Problem& p) { return p.cu_seqlens ? p.nseq : p.B; }

// Chunks of all sequences: exact for a batch, an upper bound for packed
// sequences (sum of ceil(len / C) <= ceil(T / C) + nseq).
inline long max_chunks(const Problem& p) {
  return p.cu_seqlens ? (long)p.N + p.nseq : (long)p.B * p.N;
}

// Device view of the sequences of a call, shared by every kernel.  Tokens
// live in [B, T, H, D] tensors; a sequence is addressed by its batch row b
// and first token t0 within it, its length and chunk count, and the global
// index of per-chunk records (T tiles, entry states), laid out
// [chunk][head] for packed sequences and [sequence * H + head][chunk] for a
// batch.
struct Seqs {
  const int* cu;     // packed: [nseq + 1] token offsets; nullptr: a batch
  const int* choff;  // packed: [nseq + 1] chunk offsets
  int T, N, H, C;    // batch: tokens and chunks per row; heads; chunk size

  __host__ __device__ static Seqs of(const Problem& p) {
    return Seqs{p.cu_seqlens, p.chunk_off, p.T, p.N, p.H, p.C};
  }
  // batch row, first token within it, length and chunks of sequence s
  __device__ __forceinline__ void get(int s, int& b, int& t0, int& len, int& nch) const {
    if (!cu) {
      b = s, t0 = 0, len = T, nch = N;
    } else {  // chunk counts from the offsets: all zero when cu_seqlens was invalid
      b = 0, t0 = cu[s], len = cu[s + 1] - cu[s], nch = choff[s + 1] - choff[s];
    }
  }
  // index of the per-chunk record of chunk ci of (sequence s, head h)
  __device__ __forceinline__ size_t rec(int s, int h, int ci) const {
    return cu ? (size_t)(choff[s] + ci) * H + h : ((size_t)s * H + h) * N + ci;
  }
  // the same with the mode fixed at compile time (kernels instantiated per mode)
  template <bool Packed>
  __device__ __forceinline__ void get_t(int s, int& b, int& t0, int& len, int& nch) const {
    if constexpr (Packed) {
      b = 0, t0 = cu[s], len = cu[s + 1] - cu[s], nch = choff[s + 1] - choff[s];
    } else {
      b = s, t0 = 0, len = T, nch = N;
    }
  }
  template <bool Packed>
  __device__ __forceinline__ size_t rec_t(int s, int h, int ci) const {
    if constexpr (Packed) return (size_t)(choff[s] + ci) * H + h;
    else return (size_t)(s * H + h) * N + ci;
  }
  // chunk-parallel kernels: the (sequence, head, chunk) of block x of a grid
  // of max_chunks * H blocks; false for blocks past the last chunk
  __device__ __forceinline__ bool chunk_of(long x, int nseq, int& s, int& h, int& ci) const {
    if (!cu) {
      const long bh = x / N;
      ci = (int)(x % N), s = (int)(bh / H), h = (int)(bh % H);
      return true;
    }
    const long gc = x / H;
    h = (int)(x % H);
    if (gc >= choff[nseq]) return false;
    int lo = 0, hi = nseq - 1;  // the last s with choff[s] <= gc
    while (lo < hi) {
      const int mid = (lo + hi + 1) / 2;
      if (choff[mid] <= gc) lo = mid;
      else hi = mid - 1;
    }
    s = lo, ci = (int)(gc - choff[lo]);
    return true;
  }
};

// Record index of chunk ci for a kernel whose block is bh = s * H + h (for a
// batch simply bh * N + ci, N the chunks per sequence).
template <bool Packed>
__device__ __forceinline__ size_t rec_bh(const Seqs& q, int N, int bh, int s, int h, int ci) {
  if constexpr (Packed) return q.template rec_t<true>(s, h, ci);
  else return (size_t)bh * N + ci;
}

// Packed sequences: checks cu_seqlens (non-decreasing from 0 to T) and writes
// the chunk offsets; an invalid offset array is recorded as
// GDN_ERR_SEQLENS in the device status word and leaves every chunk count at
// zero, so that the kernels that follow do nothing.
cudaError_t setup_seqlens(const Problem& p, int* chunk_off, cudaStream_t s);

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

// The mixer's fused neighbours (neighbours.cu).  Short convolution over
// x [B, T, H*D] (packed: B = 1 and cu_seqlens/nseq as for the mixer) with
// weights w [H*D, W]; gated RMS norm over rows of D values.
struct ConvProblem {
  int B = 0, T = 0, H = 0, D = 0, W = 0;
  bool bf16 = true, l2norm = false;
  float scale = 1.f, eps = 1e-6f;
  const int* cu_seqlens = nullptr;
  int nseq = 0;
  const void* x = nullptr;
  const float* w = nullptr;
  void* z = nullptr;
  const void* dz = nullptr;
  void* dx = nullptr;
  float* dw = nullptr;
  void* ws = nullptr;
};
size_t short_conv_bwd_workspace(const ConvProblem& p);
cudaError_t short_conv_fwd(const ConvProblem& p, cudaStream_t s);
cudaError_t short_conv_bwd(const ConvProblem& p, cudaStream_t s);

struct NormProblem {
  long rows = 0;
  int D = 0;
  bool bf16 = true;
  float eps = 1e-6f;
  const void* o = nullptr;
  const void* gate = nullptr;
  const float* weight = nullptr;
  void* out = nullptr;
  const void* dout = nullptr;
  void* dO = nullptr;
  void* dgate = nullptr;
  float* dweight = nullptr;
  void* ws = nullptr;
};
size_t gated_rmsnorm_bwd_workspace(const NormProblem& p);
cudaError_t gated_rmsnorm_fwd(const NormProblem& p, cudaStream_t s);
cudaError_t gated_rmsnorm_bwd(const NormProblem& p, cudaStream_t s);
cudaError_t nb_read_and_clear_status(int* status);

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
  kSeqSetup = 15,
  kConvFwd = 16,
  kConvBwd = 17,
  kNormFwd = 18,
  kNormBwd = 19,
  kSumPartials = 20,
  kNumKernelIds = 21
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
