// C ABI of the GDN / KDA mixer: argument checks, kernel selection, launch.
// The operations, layouts and error rules are stated in include/gdn.h.

#include <initializer_list>
#include <vector>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace {

struct ProfileState {
  bool on = false;
  int cap = 0, n = 0, launches = 0;
  std::vector<cudaEvent_t> ev;  // 2 per recorded launch
  std::vector<int> ids;
};
thread_local ProfileState g_prof;

thread_local int g_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = (int)e;
  return GDN_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Validates the shape; fills the size fields of a Problem.
int check_shape(const gdn_shape* s, bool kda, gdn::Problem* p, bool no_delta = false) {
  if (!s) return GDN_ERR_ARG;
  if (s->dtype != GDN_F32 && s->dtype != GDN_BF16 && !(kda && s->dtype == GDN_BF16_G16))
    return GDN_ERR_DTYPE;
  if (s->B < 0 || s->T < 0 || s->H < 0) return GDN_ERR_SHAPE;
  if (s->dk < 1 || s->dk > 128 || s->dv < 1 || s->dv > 128) return GDN_ERR_SHAPE;
  if (s->chunk != 16 && s->chunk != 32 && s->chunk != 64) return GDN_ERR_SHAPE;
  *p = gdn::Problem{};
  p->B = s->B;
  p->T = s->T;
  p->H = s->H;
  p->dk = s->dk;
  p->dv = s->dv;
  p->C = s->chunk;
  p->N = (s->T + s->chunk - 1) / s->chunk;
  p->kda = kda;
  p->no_delta = no_delta;
  p->bf16 = s->dtype == GDN_BF16 || s->dtype == GDN_BF16_G16;
  p->g16 = s->dtype == GDN_BF16_G16;
  return GDN_OK;
}

bool empty(const gdn::Problem& p) { return gdn::num_seqs(p) == 0 || p.H == 0; }

// Packed sequences: the chunk offsets sit in front of the mixer's workspace.
size_t seq_prefix(const gdn::Problem& p) {
  return p.cu_seqlens ? gdn::align_up((size_t)(p.nseq + 1) * sizeof(int), 256) : 0;
}

// Marks a problem as packed (B must be 1); the pointer is the caller's
// device array of nseq + 1 token offsets.
int set_packed(gdn::Problem* p, const int* cu_seqlens, int nseq) {
  if (nseq < 0) return GDN_ERR_SHAPE;
  if (p->B != 1) return GDN_ERR_SHAPE;
  if (!cu_seqlens) return GDN_ERR_ARG;
  if (((uintptr_t)cu_seqlens & 3u) != 0) return GDN_ERR_ALIGN;
  p->cu_seqlens = cu_seqlens;
  p->nseq = nseq;
  return GDN_OK;
}

size_t fwd_ws(const gdn::Problem& p) {
  if (empty(p) || p.T == 0) return 0;
  if (gdn::kda_tc_supported(p)) return gdn::kda_tc_fwd_workspace(p);
  return gdn::tc_supported(p) ? gdn::tc_fwd_workspace(p) : 0;
}

size_t bwd_ws(const gdn::Problem& p) {
  if (empty(p) || p.T == 0) return 0;
  if (gdn::kda_tc_supported(p)) return gdn::kda_tc_bwd_workspace(p);
  return gdn::tc_supported(p) ? gdn::tc_bwd_workspace(p) : gdn::simt_bwd_workspace(p);
}

// The CUDA-core path's context is the backward pass's workspace, whose first
// part (the fp32 entry state of every chunk) the forward pass fills; the KDA
// tensor-core path's is its backward workspace as well.
size_t ctx_bytes(const gdn::Problem& p) {
  if (empty(p) || p.T == 0) return 0;
  if (gdn::kda_tc_supported(p)) return gdn::kda_tc_bwd_workspace(p);
  return gdn::tc_supported(p) ? gdn::tc_ctx_bytes(p) : gdn::simt_bwd_workspace(p);
}

// Zero-length sequences: the final state is the initial one and every
// gradient of the (empty) token tensors is empty.
cudaError_t copy_state_or_zero(float* dst, const float* src, const gdn::Problem& p,
                               cudaStream_t st) {
  const size_t bytes = (size_t)gdn::num_seqs(p) * p.H * p.dk * p.dv * sizeof(float);
  if (!dst) return cudaSuccess;
  if (src) return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice, st);
  return cudaMemsetAsync(dst, 0, bytes, st);
}

int run_fwd(const gdn_shape* shape, bool kda, const void* q, const void* k, const void* v,
            const void* g, const float* beta, const float* h0, void* o, float* ht, void* ws,
            size_t ws_bytes, void* stream, bool save = false, bool no_delta = false,
            const int* cu_seqlens = nullptr, int nseq = -1) {
  gdn::Problem p;
  int rc = check_shape(shape, kda, &p, no_delta);
  if (rc != GDN_OK) return rc;
  if (nseq >= 0 && (rc = set_packed(&p, cu_seqlens, nseq)) != GDN_OK) return rc;
  if (empty(p)) return GDN_OK;
  // token tensors of an empty sequence hold no data and may be NULL
  if (p.T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, h0, o, ht, ws};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return GDN_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.T == 0) {
    cudaError_t e = copy_state_or_zero(ht, h0, p, st);
    return e == cudaSuccess ? GDN_OK : fail_cuda(e);
  }
  const size_t pre = seq_prefix(p);
  const size_t need = pre + (save ? ctx_bytes(p) : fwd_ws(p));
  if (need > 0 && (!ws || ws_bytes < need)) return GDN_ERR_WORKSPACE;
  p.q = q; p.k = k; p.v = v; p.g = static_cast<const float*>(g); p.beta = beta; p.h0 = h0; p.o = o; p.ht = ht;
  p.ws = static_cast<unsigned char*>(ws) + pre;
  p.ws_bytes = ws_bytes - pre;
  if (p.cu_seqlens) {
    p.chunk_off = static_cast<int*>(ws);
    cudaError_t e = gdn::setup_seqlens(p, static_cast<int*>(ws), st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  cudaError_t e = gdn::kda_tc_supported(p) ? gdn::kda_tc_fwd(p, st, save)
                  : gdn::tc_supported(p)     ? gdn::tc_fwd(p, st, save)
                                             : gdn::simt_fwd(p, st, save);
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

int run_bwd(const gdn_shape* shape, bool kda, const void* q, const void* k, const void* v,
            const void* g, const float* beta, const float* h0, const void* do_,
            const float* dht, void* dq, void* dk, void* dv, void* dg, float* dbeta,
            float* dh0, void* ws, size_t ws_bytes, void* stream, bool saved = false,
            bool no_delta = false, const int* cu_seqlens = nullptr, int nseq = -1) {
  gdn::Problem p;
  int rc = check_shape(shape, kda, &p, no_delta);
  if (rc != GDN_OK) return rc;
  if (nseq >= 0 && (rc = set_packed(&p, cu_seqlens, nseq)) != GDN_OK) return rc;
  if (empty(p)) return GDN_OK;
  if (p.T > 0 && (!q || !k || !v || !g || !beta || !do_ || !dq || !dk || !dv || !dg || !dbeta))
    return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ws};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return GDN_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.T == 0) {
    cudaError_t e = copy_state_or_zero(dh0, dht, p, st);
    return e == cudaSuccess ? GDN_OK : fail_cuda(e);
  }
  const size_t pre = seq_prefix(p);
  const size_t need = pre + (saved ? ctx_bytes(p) : bwd_ws(p));
  if (need > 0 && (!ws || ws_bytes < need)) return GDN_ERR_WORKSPACE;
  p.q = q; p.k = k; p.v = v; p.g = static_cast<const float*>(g); p.beta = beta; p.h0 = h0; p.do_ = do_; p.dht = dht;
  p.dq = dq; p.dk_ = dk; p.dv_ = dv; p.dg = static_cast<float*>(dg); p.dbeta = dbeta; p.dh0 = dh0;
  p.ws = static_cast<unsigned char*>(ws) + pre;
  p.ws_bytes = ws_bytes - pre;
  if (p.cu_seqlens) {
    p.chunk_off = static_cast<int*>(ws);
    cudaError_t e = gdn::setup_seqlens(p, static_cast<int*>(ws), st);
    if (e != cudaSuccess) return fail_cuda(e);
  }
  cudaError_t e = gdn::kda_tc_supported(p) ? gdn::kda_tc_bwd(p, st, saved)
                  : gdn::tc_supported(p)     ? gdn::tc_bwd(p, st, saved)
                                             : gdn::simt_bwd(p, st, saved);
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

int run_decode(const gdn_shape* shape, bool kda, const void* q, const void* k, const void* v,
               const void* g, const float* beta, const float* h0, void* o, float* ht,
               void* stream) {
  gdn::Problem p;
  int rc = check_shape(shape, kda, &p);
  if (rc != GDN_OK) return rc;
  if (empty(p)) return GDN_OK;
  if (p.T > 0 && (!q || !k || !v || !g || !beta || !o)) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, h0, o, ht};
  for (const void* x : ptrs)
    if (x && !aligned16(x)) return GDN_ERR_ALIGN;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.T == 0) {
    if (ht == h0 && ht) return GDN_OK;  // in place: nothing changes
    cudaError_t e = copy_state_or_zero(ht, h0, p, st);
    return e == cudaSuccess ? GDN_OK : fail_cuda(e);
  }
  p.q = q; p.k = k; p.v = v; p.g = static_cast<const float*>(g); p.beta = beta; p.h0 = h0; p.o = o; p.ht = ht;
  cudaError_t e = gdn::decode(p, st);
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

size_t query_ws(const gdn_shape* shape, bool kda, bool bwd, bool no_delta = false, int nseq = -1) {
  gdn::Problem p;
  if (check_shape(shape, kda, &p, no_delta) != GDN_OK) return 0;
  static const int kAnyOffsets[1] = {0};  // only the size matters here
  if (nseq >= 0 && set_packed(&p, kAnyOffsets, nseq) != GDN_OK) return 0;
  if (empty(p) || p.T == 0) return 0;
  return seq_prefix(p) + (bwd ? bwd_ws(p) : fwd_ws(p));
}

size_t query_ctx(const gdn_shape* shape, bool kda, bool no_delta = false) {
  gdn::Problem p;
  if (check_shape(shape, kda, &p, no_delta) != GDN_OK) return 0;
  return ctx_bytes(p);
}

}  // namespace

namespace gdn {

int record_cuda_error(cudaError_t e) { return fail_cuda(e); }

const char* kernel_name(int id) {
  static const char* names[kNumKernelIds] = {
      "simt_fwd", "simt_states", "simt_bwd", "simt_bwd_reduce",
      "tc_fwd", "tc_states", "tc_bwd", "tc_solve", "tc_fwd_segment", "tc_combine", "decode",
      "kda_tc_prep", "kda_tc_fwd", "kda_tc_states", "kda_tc_bwd", "seqlens_setup",
      "short_conv_fwd", "short_conv_bwd", "gated_rmsnorm_fwd", "gated_rmsnorm_bwd", "sum_partials"};
  return (id >= 0 && id < kNumKernelIds) ? names[id] : "unknown";
}

void prof_before(cudaStream_t s) {
  ProfileState& P = g_prof;
  if (P.on && P.n < P.cap) cudaEventRecord(P.ev[2 * P.n], s);
}

void prof_after(cudaStream_t s, int kernel_id) {
  ProfileState& P = g_prof;
  if (!P.on) return;
  if (P.n < P.cap) {
    cudaEventRecord(P.ev[2 * P.n + 1], s);
    P.ids[P.n] = kernel_id;
    ++P.n;
  }
  ++P.launches;
}

}  // namespace gdn

extern "C" {

int gdn_profile_begin(int cap) {
  ProfileState& P = g_prof;
  if (cap < 0) return GDN_ERR_ARG;
  while ((int)P.ev.size() < 2 * cap) {
    cudaEvent_t e;
    cudaError_t err = cudaEventCreate(&e);
    if (err != cudaSuccess) return fail_cuda(err);
    P.ev.push_back(e);
  }
  P.ids.assign(cap, -1);
  P.cap = cap;
  P.n = 0;
  P.launches = 0;
  P.on = true;
  return GDN_OK;
}

int gdn_profile_end(void) {
  g_prof.on = false;
  return g_prof.launches;
}

int gdn_profile_read(int* kernel_ids, float* ms, int max) {
  ProfileState& P = g_prof;
  const int n = P.n < max ? P.n : max;
  for (int i = 0; i < n; ++i) {
    cudaError_t e = cudaEventSynchronize(P.ev[2 * i + 1]);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&ms[i], P.ev[2 * i], P.ev[2 * i + 1]);
    if (e != cudaSuccess) return fail_cuda(e);
    kernel_ids[i] = P.ids[i];
  }
  return n;
}

const char* gdn_kernel_name(int kernel_id) { return gdn::kernel_name(kernel_id); }

size_t gdn_fwd_workspace(const gdn_shape* shape) { return query_ws(shape, false, false); }
size_t kda_fwd_workspace(const gdn_shape* shape) { return query_ws(shape, true, false); }
size_t gdn_bwd_workspace(const gdn_shape* shape) { return query_ws(shape, false, true); }
size_t kda_bwd_workspace(const gdn_shape* shape) { return query_ws(shape, true, true); }

int gdn_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v, const float* g,
            const float* beta, const float* h0, void* o, float* ht, void* ws, size_t ws_bytes,
            void* stream) {
  return run_fwd(shape, false, q, k, v, g, beta, h0, o, ht, ws, ws_bytes, stream);
}

int kda_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v, const void* g,
            const float* beta, const float* h0, void* o, float* ht, void* ws, size_t ws_bytes,
            void* stream) {
  return run_fwd(shape, true, q, k, v, g, beta, h0, o, ht, ws, ws_bytes, stream);
}

int gdn_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v, const float* g,
            const float* beta, const float* h0, const void* do_, const float* dht, void* dq,
            void* dk, void* dv, float* dg, float* dbeta, float* dh0, void* ws, size_t ws_bytes,
            void* stream) {
  return run_bwd(shape, false, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ws,
                 ws_bytes, stream);
}

int kda_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v, const void* g,
            const float* beta, const float* h0, const void* do_, const float* dht, void* dq,
            void* dk, void* dv, void* dg, float* dbeta, float* dh0, void* ws, size_t ws_bytes,
            void* stream) {
  return run_bwd(shape, true, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ws,
                 ws_bytes, stream);
}

size_t gdn_ctx_bytes(const gdn_shape* shape) { return query_ctx(shape, false); }
size_t kda_ctx_bytes(const gdn_shape* shape) { return query_ctx(shape, true); }

int gdn_fwd_save(const gdn_shape* shape, const void* q, const void* k, const void* v,
                 const float* g, const float* beta, const float* h0, void* o, float* ht,
                 void* ctx, size_t ctx_bytes, void* stream) {
  return run_fwd(shape, false, q, k, v, g, beta, h0, o, ht, ctx, ctx_bytes, stream, true);
}

int kda_fwd_save(const gdn_shape* shape, const void* q, const void* k, const void* v,
                 const void* g, const float* beta, const float* h0, void* o, float* ht,
                 void* ctx, size_t ctx_bytes, void* stream) {
  return run_fwd(shape, true, q, k, v, g, beta, h0, o, ht, ctx, ctx_bytes, stream, true);
}

int gdn_bwd_saved(const gdn_shape* shape, const void* q, const void* k, const void* v,
                  const float* g, const float* beta, const float* h0, const void* do_,
                  const float* dht, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                  float* dh0, void* ctx, size_t ctx_bytes, void* stream) {
  return run_bwd(shape, false, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ctx,
                 ctx_bytes, stream, true);
}

int kda_bwd_saved(const gdn_shape* shape, const void* q, const void* k, const void* v,
                  const void* g, const float* beta, const float* h0, const void* do_,
                  const float* dht, void* dq, void* dk, void* dv, void* dg, float* dbeta,
                  float* dh0, void* ctx, size_t ctx_bytes, void* stream) {
  return run_bwd(shape, true, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ctx,
                 ctx_bytes, stream, true);
}

int gdn_decode(const gdn_shape* shape, const void* q, const void* k, const void* v,
               const float* g, const float* beta, const float* h0, void* o, float* ht,
               void* stream) {
  return run_decode(shape, false, q, k, v, g, beta, h0, o, ht, stream);
}

int kda_decode(const gdn_shape* shape, const void* q, const void* k, const void* v,
               const void* g, const float* beta, const float* h0, void* o, float* ht,
               void* stream) {
  return run_decode(shape, true, q, k, v, g, beta, h0, o, ht, stream);
}

size_t mamba2_fwd_workspace(const gdn_shape* shape) { return query_ws(shape, false, false, true); }
size_t mamba2_bwd_workspace(const gdn_shape* shape) { return query_ws(shape, false, true, true); }
size_t mamba2_ctx_bytes(const gdn_shape* shape) { return query_ctx(shape, false, true); }

int mamba2_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
               const float* g, const float* beta, const float* h0, void* o, float* ht, void* ws,
               size_t ws_bytes, void* stream) {
  return run_fwd(shape, false, q, k, v, g, beta, h0, o, ht, ws, ws_bytes, stream, false, true);
}

int mamba2_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
               const float* g, const float* beta, const float* h0, const void* do_,
               const float* dht, void* dq, void* dk, void* dv, float* dg, float* dbeta,
               float* dh0, void* ws, size_t ws_bytes, void* stream) {
  return run_bwd(shape, false, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ws,
                 ws_bytes, stream, false, true);
}

int mamba2_fwd_save(const gdn_shape* shape, const void* q, const void* k, const void* v,
                    const float* g, const float* beta, const float* h0, void* o, float* ht,
                    void* ctx, size_t ctx_bytes, void* stream) {
  return run_fwd(shape, false, q, k, v, g, beta, h0, o, ht, ctx, ctx_bytes, stream, true, true);
}

int mamba2_bwd_saved(const gdn_shape* shape, const void* q, const void* k, const void* v,
                     const float* g, const float* beta, const float* h0, const void* do_,
                     const float* dht, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                     float* dh0, void* ctx, size_t ctx_bytes, void* stream) {
  return run_bwd(shape, false, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ctx,
                 ctx_bytes, stream, true, true);
}

size_t gdn_varlen_workspace(const gdn_shape* shape, int nseq, int backward) {
  return query_ws(shape, false, backward != 0, false, nseq);
}
size_t kda_varlen_workspace(const gdn_shape* shape, int nseq, int backward) {
  return query_ws(shape, true, backward != 0, false, nseq);
}
size_t mamba2_varlen_workspace(const gdn_shape* shape, int nseq, int backward) {
  return query_ws(shape, false, backward != 0, true, nseq);
}

#define GDN_VARLEN_PAIR(name, kda, nodelta, GT, DGT)                                               \
  int name##_fwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq, const void* q,  \
                        const void* k, const void* v, const GT* g, const float* beta,            \
                        const float* h0, void* o, float* ht, void* ws, size_t ws_bytes,          \
                        void* stream) {                                                          \
    if (nseq < 0) return GDN_ERR_SHAPE;                                                          \
    return run_fwd(shape, kda, q, k, v, g, beta, h0, o, ht, ws, ws_bytes, stream, false,         \
                   nodelta, cu_seqlens, nseq);                                                    \
  }                                                                                              \
  int name##_bwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq, const void* q,  \
                        const void* k, const void* v, const GT* g, const float* beta,            \
                        const float* h0, const void* do_, const float* dht, void* dq, void* dk,  \
                        void* dv, DGT* dg, float* dbeta, float* dh0, void* ws,                   \
                        size_t ws_bytes, void* stream) {                                         \
    if (nseq < 0) return GDN_ERR_SHAPE;                                                          \
    return run_bwd(shape, kda, q, k, v, g, beta, h0, do_, dht, dq, dk, dv, dg, dbeta, dh0, ws,   \
                   ws_bytes, stream, false, nodelta, cu_seqlens, nseq);                           \
  }
GDN_VARLEN_PAIR(gdn, false, false, float, float)
GDN_VARLEN_PAIR(kda, true, false, void, void)  // fp32 or bf16 gate (GDN_BF16_G16)
GDN_VARLEN_PAIR(mamba2, false, true, float, float)
#undef GDN_VARLEN_PAIR

}  // extern "C"

// ---------------------------------------------------------------- neighbours
namespace {

int conv_problem(const gdn_conv_shape* s, int l2norm, float scale, float eps,
                 const int* cu_seqlens, int nseq, gdn::ConvProblem* p) {
  if (!s) return GDN_ERR_ARG;
  if (s->dtype != GDN_F32 && s->dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (s->B < 0 || s->T < 0 || s->H < 0) return GDN_ERR_SHAPE;
  if (s->D != 32 && s->D != 64 && s->D != 128) return GDN_ERR_SHAPE;
  if (s->W < 1 || s->W > 4) return GDN_ERR_SHAPE;
  if (!(eps >= 0.f)) return GDN_ERR_ARG;
  if (s->H > 65535 || (long long)s->H * s->D > (1 << 24)) return GDN_ERR_SHAPE;
  if ((long long)s->B * s->T > (1LL << 30)) return GDN_ERR_SHAPE;
  *p = gdn::ConvProblem{};
  p->B = s->B; p->T = s->T; p->H = s->H; p->D = s->D; p->W = s->W;
  p->bf16 = s->dtype == GDN_BF16;
  p->l2norm = l2norm != 0;
  p->scale = scale;
  p->eps = eps;
  if (cu_seqlens) {
    if (s->B != 1 || nseq < 0) return GDN_ERR_SHAPE;
    if (((uintptr_t)cu_seqlens & 3u) != 0) return GDN_ERR_ALIGN;
    p->cu_seqlens = cu_seqlens;
    p->nseq = nseq;
  }
  return GDN_OK;
}

bool conv_empty(const gdn::ConvProblem& p) { return (long long)p.B * p.T == 0 || p.H == 0; }

int norm_problem(const gdn_norm_shape* s, float eps, gdn::NormProblem* p) {
  if (!s) return GDN_ERR_ARG;
  if (s->dtype != GDN_F32 && s->dtype != GDN_BF16) return GDN_ERR_DTYPE;
  if (s->rows < 0) return GDN_ERR_SHAPE;
  if (s->D != 32 && s->D != 64 && s->D != 128) return GDN_ERR_SHAPE;
  if (!(eps >= 0.f)) return GDN_ERR_ARG;
  *p = gdn::NormProblem{};
  p->rows = (long)s->rows;
  p->D = s->D;
  p->bf16 = s->dtype == GDN_BF16;
  p->eps = eps;
  return GDN_OK;
}

bool all_aligned(std::initializer_list<const void*> ptrs) {
  for (const void* x : ptrs)
    if (!x || !aligned16(x)) return false;
  return true;
}

bool any_null(std::initializer_list<const void*> ptrs) {
  for (const void* x : ptrs)
    if (!x) return true;
  return false;
}

}  // namespace

extern "C" {

int gdn_short_conv_fwd(const gdn_conv_shape* shape, const void* x, const float* w, void* z,
                       int l2norm, float scale, float eps, const int* cu_seqlens, int nseq,
                       void* stream) {
  gdn::ConvProblem p;
  int rc = conv_problem(shape, l2norm, scale, eps, cu_seqlens, nseq, &p);
  if (rc != GDN_OK || conv_empty(p)) return rc;
  if (any_null({x, w, z})) return GDN_ERR_ARG;
  if (!all_aligned({x, z})) return GDN_ERR_ALIGN;
  p.x = x; p.w = w; p.z = z;
  cudaError_t e = gdn::short_conv_fwd(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

size_t gdn_short_conv_bwd_workspace(const gdn_conv_shape* shape) {
  gdn::ConvProblem p;
  if (conv_problem(shape, 0, 1.f, 0.f, nullptr, 0, &p) != GDN_OK) return 0;
  return gdn::short_conv_bwd_workspace(p);
}

int gdn_short_conv_bwd(const gdn_conv_shape* shape, const void* x, const float* w,
                       const void* dz, void* dx, float* dw, int l2norm, float scale, float eps,
                       const int* cu_seqlens, int nseq, void* ws, size_t ws_bytes,
                       void* stream) {
  gdn::ConvProblem p;
  int rc = conv_problem(shape, l2norm, scale, eps, cu_seqlens, nseq, &p);
  if (rc != GDN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (conv_empty(p)) {
    // no token: dw is the empty sum
    if (!dw) return GDN_ERR_ARG;
    const size_t n = (size_t)p.H * p.D * p.W;
    cudaError_t e = n ? cudaMemsetAsync(dw, 0, n * sizeof(float), st) : cudaSuccess;
    return e == cudaSuccess ? GDN_OK : fail_cuda(e);
  }
  if (any_null({x, w, dz, dx, dw})) return GDN_ERR_ARG;
  if (!all_aligned({x, dz, dx})) return GDN_ERR_ALIGN;
  const size_t need = gdn::short_conv_bwd_workspace(p);
  if (!ws || ws_bytes < need) return GDN_ERR_WORKSPACE;
  if (!aligned16(ws)) return GDN_ERR_ALIGN;
  p.x = x; p.w = w; p.dz = dz; p.dx = dx; p.dw = dw; p.ws = ws;
  cudaError_t e = gdn::short_conv_bwd(p, st);
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

int gdn_gated_rmsnorm_fwd(const gdn_norm_shape* shape, const void* o, const void* gate,
                          const float* weight, void* out, float eps, void* stream) {
  gdn::NormProblem p;
  int rc = norm_problem(shape, eps, &p);
  if (rc != GDN_OK || p.rows == 0) return rc;
  if (any_null({o, gate, weight, out})) return GDN_ERR_ARG;
  if (!all_aligned({o, gate, out})) return GDN_ERR_ALIGN;
  p.o = o; p.gate = gate; p.weight = weight; p.out = out;
  cudaError_t e = gdn::gated_rmsnorm_fwd(p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

size_t gdn_gated_rmsnorm_bwd_workspace(const gdn_norm_shape* shape) {
  gdn::NormProblem p;
  if (norm_problem(shape, 0.f, &p) != GDN_OK) return 0;
  return gdn::gated_rmsnorm_bwd_workspace(p);
}

int gdn_gated_rmsnorm_bwd(const gdn_norm_shape* shape, const void* o, const void* gate,
                          const float* weight, const void* dout, void* do_, void* dgate,
                          float* dweight, float eps, void* ws, size_t ws_bytes, void* stream) {
  gdn::NormProblem p;
  int rc = norm_problem(shape, eps, &p);
  if (rc != GDN_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (p.rows == 0) {
    if (!dweight) return GDN_ERR_ARG;
    cudaError_t e = cudaMemsetAsync(dweight, 0, (size_t)p.D * sizeof(float), st);
    return e == cudaSuccess ? GDN_OK : fail_cuda(e);
  }
  if (any_null({o, gate, weight, dout, do_, dgate, dweight})) return GDN_ERR_ARG;
  if (!all_aligned({o, gate, dout, do_, dgate})) return GDN_ERR_ALIGN;
  const size_t need = gdn::gated_rmsnorm_bwd_workspace(p);
  if (!ws || ws_bytes < need) return GDN_ERR_WORKSPACE;
  if (!aligned16(ws)) return GDN_ERR_ALIGN;
  p.o = o; p.gate = gate; p.weight = weight; p.dout = dout; p.dO = do_; p.dgate = dgate;
  p.dweight = dweight; p.ws = ws;
  cudaError_t e = gdn::gated_rmsnorm_bwd(p, st);
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

const char* gdn_status_str(int status) {
  switch (status) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_ARG: return "GDN_ERR_ARG: a required pointer is NULL";
    case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE: invalid B/T/H, head dimension or chunk size";
    case GDN_ERR_DTYPE: return "GDN_ERR_DTYPE: dtype must be GDN_F32 or GDN_BF16";
    case GDN_ERR_ALIGN: return "GDN_ERR_ALIGN: pointers must be 16-byte aligned";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE: workspace missing or too small";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA: a CUDA call failed (see gdn_last_cuda_error)";
    case GDN_ERR_DEVICE_TIMEOUT: return "GDN_ERR_DEVICE_TIMEOUT: a device-side wait ran out";
    case GDN_ERR_SEQLENS:
      return "GDN_ERR_SEQLENS: cu_seqlens does not rise from 0 to T (packed sequences)";
    default: return "unknown gdn_status";
  }
}

int gdn_last_cuda_error(void) { return g_last_cuda_error; }

int gdn_device_status(void) {
  int status = GDN_OK;
  cudaError_t e = gdn::read_and_clear_device_status(&status);
  if (e != cudaSuccess) return fail_cuda(e);
  return status;
}

int gdn_wait_selftest(int max_tries, void* stream) {
  if (max_tries < 1 || max_tries > 1000) return GDN_ERR_ARG;
  cudaError_t e = gdn::wait_selftest(max_tries, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GDN_OK : fail_cuda(e);
}

int gdn_uses_tensor_cores(const gdn_shape* shape) {
  gdn::Problem p;
  if (check_shape(shape, false, &p) != GDN_OK) return 0;
  return gdn::tc_supported(p) ? 1 : 0;
}

int kda_uses_tensor_cores(const gdn_shape* shape) {
  gdn::Problem p;
  if (check_shape(shape, true, &p) != GDN_OK) return 0;
  return gdn::kda_tc_supported(p) ? 1 : 0;
}

}  // extern "C"
