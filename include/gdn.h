/*
 * gdn.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet / Kimi Delta Attention
 * token mixer, forward and backward.
 *
 * The operation.  The Primus hybrid-LLM pretraining blog (MI355X), section
 * "How hybrid models are defined in Primus", names the two linear-recurrent
 * mixers built here: Gated DeltaNet (GDN), which adds the delta rule -- the
 * state rewrites the value stored under the current key rather than only
 * accumulating -- to a state with one scalar forget gate per head, and Kimi
 * Delta Attention (KDA), which refines that gate to one value per key
 * dimension.  Per batch row b and head h, over tokens t, with the state kept
 * as H (dk x dv, fp32; H = S^T of the usual S_t = a_t S_{t-1}(I - b_t k_t
 * k_t^T) + b_t v_t k_t^T, o_t = S_t q_t):
 *
 *   GDN:  H_t = exp(g_t) (I - beta_t k_t k_t^T) H_{t-1} + beta_t k_t v_t^T
 *   KDA:  H_t = (I - beta_t k_t k_t^T) diag(exp(g_t)) H_{t-1} + beta_t k_t v_t^T
 *   o_t = H_t^T q_t,   H_{-1} = initial state (or 0),   final state = H_{T-1}.
 *
 * The backward entry points return the gradients of a scalar loss with
 * respect to q, k, v, g, beta and the initial state, given dL/do and
 * (optionally) dL/d(final state).  They take the forward inputs again and
 * recompute what they need; no context is saved between calls.  The
 * *_fwd_save / *_bwd_saved pair below is the same computation with the
 * forward pass keeping, in a caller-owned buffer, what the backward pass
 * would otherwise recompute.
 *
 * Layout (all row-major, innermost dimension contiguous):
 *   q, k, dq, dk          [B, T, H, dk]   dtype per gdn_shape.dtype
 *   v, o, do_, dv         [B, T, H, dv]   dtype per gdn_shape.dtype
 *   g, dg (GDN)           [B, T, H]       fp32, log forget gate (a = exp(g))
 *   g, dg (KDA)           [B, T, H, dk]   fp32, or bf16 with GDN_BF16_G16
 *   beta, dbeta           [B, T, H]       fp32, used as given
 *   h0, ht, dht, dh0      [B, H, dk, dv]  fp32
 * No query scale and no normalisation is applied inside: gradients are with
 * respect to the tensors passed.
 *
 * Memory and streams.  Every pointer is a device pointer owned by the
 * caller and must be 16-byte aligned.  The library allocates nothing: each
 * pass needs a caller-provided device workspace of at least
 * *_fwd_workspace() / *_bwd_workspace() bytes (0 for some shapes, where
 * NULL/0 may be passed).  The workspace holds per-chunk intermediates of one
 * call; its contents need no initialisation and are not meaningful
 * afterwards, and two calls in flight at once need separate workspaces (the
 * saved-context pair below passes its buffer from the forward call to the
 * backward one instead; decode needs no workspace).  All
 * work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 * stream); the calls do not synchronise.  Outputs are overwritten, never
 * accumulated.  Results are deterministic (no atomics).
 *
 * Errors.  Arguments are validated on the host before anything is launched;
 * a failed check returns a negative gdn_status and launches nothing.  A
 * launch failure returns GDN_ERR_CUDA; gdn_last_cuda_error() then gives the
 * cudaError_t value.  Device-side waits are bounded: a wait that runs out
 * records GDN_ERR_DEVICE_TIMEOUT in a per-device status word that
 * gdn_device_status() reads (and clears).
 *
 * Kernel selection.  dtype BF16 with dk = dv = 128 and chunk = 64 runs the
 * tensor-core (tcgen05/TMEM, TMA-fed) kernels; every other valid shape runs
 * the CUDA-core fp32 kernels (chunk in {16, 32, 64}, 1 <= dk, dv <= 128).
 * T need not be a multiple of chunk.  KDA on the tensor cores factors each
 * chunk's per-dimension decays into scaled bf16 operand tiles; a sequence
 * with a 64-token chunk whose cumulative log gate spans more than 80 in some
 * key dimension (an average decay faster than exp(-1.25) per token there) is
 * computed by the CUDA-core kernels inside the same call, so results meet the
 * same bounds for any gates.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDN_OK = 0,
  GDN_ERR_ARG = -1,            /* NULL required pointer, bad enum value        */
  GDN_ERR_SHAPE = -2,          /* B,T,H < 0, dk/dv outside [1,128], bad chunk  */
  GDN_ERR_DTYPE = -3,          /* dtype not a gdn_dtype, or GDN_BF16_G16 with a
                                  mixer other than KDA                         */
  GDN_ERR_ALIGN = -4,          /* a pointer is not 16-byte aligned             */
  GDN_ERR_WORKSPACE = -5,      /* workspace NULL or smaller than required      */
  GDN_ERR_CUDA = -6,           /* a CUDA call failed; see gdn_last_cuda_error  */
  GDN_ERR_DEVICE_TIMEOUT = -7, /* a bounded device-side wait ran out           */
  GDN_ERR_SEQLENS = -8         /* packed sequences: cu_seqlens not rising from
                                  0 to T (found on the device; see *_varlen)   */
} gdn_status;

/* GDN_BF16_G16 (KDA only): bf16 token tensors, and the per-key-dimension gate
 * g and its gradient dg in bf16 too, which halves the gate's traffic (4 dk
 * bytes per token and head in each direction otherwise).  The kernels read
 * g as bf16, compute in fp32 exactly as with an fp32 gate holding the same
 * values, and round dg to bf16 once. */
typedef enum { GDN_F32 = 0, GDN_BF16 = 1, GDN_BF16_G16 = 2 } gdn_dtype;

/* Problem shape.  dtype is the element type of q, k, v, o, do_, dq, dk, dv
 * (GDN_BF16_G16: bf16, with a bf16 KDA gate). */
typedef struct {
  int B, T, H;  /* batch, tokens per sequence, heads; each >= 0 (0 = no work) */
  int dk, dv;   /* key / value head dimension, 1..128                         */
  int chunk;    /* tokens per chunk of the chunkwise algorithm: 16, 32 or 64  */
  int dtype;    /* gdn_dtype                                                  */
} gdn_shape;

/* With T = 0 the token pointers may be NULL: the forward pass copies h0 to ht
 * (or zeroes ht), the backward pass copies dht to dh0 (or zeroes dh0).
 *
 * Workspace bytes each entry point needs for this shape (0 if the shape is
 * invalid or needs none).  The tensor-core path of the forward pass keeps the
 * chunkwise form's triangular-solve result T = (I + A)^-1 of every 64-token
 * chunk (8 KB each, bf16), and, when few long sequences make it run each
 * sequence in segments, three fp32 dk x dv states per segment; the backward
 * pass keeps the T tiles plus the bf16 state entering every chunk (32 KB
 * each).  Everything is recomputed from the inputs inside the call.  The
 * CUDA-core fp32 path needs workspace for the backward pass only.  The
 * forward's size depends on the current device's SM count. */
GDN_API size_t gdn_fwd_workspace(const gdn_shape* shape);
GDN_API size_t kda_fwd_workspace(const gdn_shape* shape);
GDN_API size_t gdn_bwd_workspace(const gdn_shape* shape);
GDN_API size_t kda_bwd_workspace(const gdn_shape* shape);

/* GDN forward: o (and ht if non-NULL) from q, k, v, g [B,T,H], beta and h0
 * (NULL = zero initial state).  ws must hold gdn_fwd_workspace() bytes. */
GDN_API int gdn_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
            const float* g, const float* beta, const float* h0, void* o, float* ht,
            void* ws, size_t ws_bytes, void* stream);

/* GDN backward: gradients with respect to every forward input.  dht may be
 * NULL (zero gradient of the final state); dh0 may be NULL (not wanted). */
GDN_API int gdn_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
            const float* g, const float* beta, const float* h0, const void* do_,
            const float* dht, void* dq, void* dk, void* dv, float* dg, float* dbeta,
            float* dh0, void* ws, size_t ws_bytes, void* stream);

/* KDA forward / backward: as GDN, with g and dg of shape [B,T,H,dk], fp32
 * (or bf16 when shape->dtype is GDN_BF16_G16; every kda_* call takes g and
 * dg as untyped pointers for that reason). */
GDN_API int kda_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
            const void* g, const float* beta, const float* h0, void* o, float* ht,
            void* ws, size_t ws_bytes, void* stream);

GDN_API int kda_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
            const void* g, const float* beta, const float* h0, const void* do_,
            const float* dht, void* dq, void* dk, void* dv, void* dg, float* dbeta,
            float* dh0, void* ws, size_t ws_bytes, void* stream);

/* Training step with a saved context.  The backward pass needs the state
 * entering every chunk and the triangular-solve result of every chunk (the
 * chunkwise form of the recurrence above); gdn_bwd recomputes both.  The
 * pair below lets the forward pass keep them instead, in a caller-owned
 * device buffer `ctx` of at least *_ctx_bytes() bytes:
 *
 *   *_fwd_save   is *_fwd (same arguments, same results) using ctx as its
 *                workspace and leaving the context in it;
 *   *_bwd_saved  is *_bwd (same arguments, same results up to rounding) using
 *                ctx as its workspace and reading the context from it instead
 *                of recomputing it.
 *
 * The caller must pass *_bwd_saved the same shape and the same q, k, v, g,
 * beta and h0 contents as the *_fwd_save that filled ctx, with ctx not
 * written in between (nor used by another call in flight); the library
 * cannot check this, and other inputs give meaningless gradients.  On the
 * tensor-core path the context holds the bf16 entry state of every chunk
 * (32 KB) and its bf16 T = (I + A)^-1 tile (8 KB), plus the forward's
 * segment scratch; on the CUDA-core path the fp32 entry state of every chunk
 * plus the backward's scratch.  The result equals *_bwd's bit for bit except
 * after a segmented tensor-core forward (few long sequences), whose later
 * segments' entry states differ by rounding.  ctx needs no initialisation.  Errors as for
 * *_fwd / *_bwd, with GDN_ERR_WORKSPACE when ctx is NULL or smaller than
 * *_ctx_bytes(); *_ctx_bytes() is 0 for an invalid shape or one with no
 * work, and depends on the current device's SM count. */
GDN_API size_t gdn_ctx_bytes(const gdn_shape* shape);
GDN_API size_t kda_ctx_bytes(const gdn_shape* shape);

GDN_API int gdn_fwd_save(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const float* g, const float* beta, const float* h0, void* o, float* ht,
                         void* ctx, size_t ctx_bytes, void* stream);

GDN_API int gdn_bwd_saved(const gdn_shape* shape, const void* q, const void* k, const void* v,
                          const float* g, const float* beta, const float* h0, const void* do_,
                          const float* dht, void* dq, void* dk, void* dv, float* dg,
                          float* dbeta, float* dh0, void* ctx, size_t ctx_bytes, void* stream);

GDN_API int kda_fwd_save(const gdn_shape* shape, const void* q, const void* k, const void* v,
                         const void* g, const float* beta, const float* h0, void* o, float* ht,
                         void* ctx, size_t ctx_bytes, void* stream);

GDN_API int kda_bwd_saved(const gdn_shape* shape, const void* q, const void* k, const void* v,
                          const void* g, const float* beta, const float* h0, const void* do_,
                          const float* dht, void* dq, void* dk, void* dv, void* dg,
                          float* dbeta, float* dh0, void* ctx, size_t ctx_bytes, void* stream);

/* Mamba2: the mixer that GDN extends with the delta rule.  The Primus blog's
 * section "How hybrid models are defined in Primus" lists it beside GDN and
 * KDA as a selective state-space model with one scalar forget gate per head,
 * and describes GDN as that model plus the delta rule; without the delta
 * rule the state only accumulates:
 *
 *   H_t = exp(g_t) H_{t-1} + beta_t k_t v_t^T,    o_t = H_t^T q_t,
 *
 * with k, v and q in the roles of the state-space model's input projection,
 * input and read-out, and beta_t the per-token write strength (its step
 * size).  Arguments, layouts (g is [B,T,H]), workspace rules, saved context,
 * errors and kernel selection are those of the gdn_* calls of the same name;
 * the chunkwise form needs no triangular solve (T = I). */
GDN_API size_t mamba2_fwd_workspace(const gdn_shape* shape);
GDN_API size_t mamba2_bwd_workspace(const gdn_shape* shape);
GDN_API size_t mamba2_ctx_bytes(const gdn_shape* shape);
GDN_API int mamba2_fwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* h0, void* o, float* ht,
                       void* ws, size_t ws_bytes, void* stream);
GDN_API int mamba2_bwd(const gdn_shape* shape, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* h0, const void* do_,
                       const float* dht, void* dq, void* dk, void* dv, float* dg, float* dbeta,
                       float* dh0, void* ws, size_t ws_bytes, void* stream);
GDN_API int mamba2_fwd_save(const gdn_shape* shape, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const float* h0, void* o,
                            float* ht, void* ctx, size_t ctx_bytes, void* stream);
GDN_API int mamba2_bwd_saved(const gdn_shape* shape, const void* q, const void* k,
                             const void* v, const float* g, const float* beta, const float* h0,
                             const void* do_, const float* dht, void* dq, void* dk, void* dv,
                             float* dg, float* dbeta, float* dh0, void* ctx, size_t ctx_bytes,
                             void* stream);

/* Packed variable-length sequences.  The *_varlen calls take nseq sequences
 * of different lengths packed one after another along the token dimension,
 * as the 1M-token SFT guide packs its samples (section 4.2): shape->B must
 * be 1 and shape->T the total token count; cu_seqlens is a DEVICE array of
 * nseq + 1 int32 token offsets (4-byte aligned), sequence s being tokens
 * [cu_seqlens[s], cu_seqlens[s+1]).  Each sequence starts from its own
 * initial state and ends in its own final state: h0, ht, dht and dh0 are
 * [nseq, H, dk, dv]; every other tensor keeps its [1, T, H, ...] layout.  A
 * sequence may be empty (its final state is its initial one).  Arguments,
 * dtypes, kernel selection and errors are those of the fixed-length calls,
 * except that the workspace is *_varlen_workspace(shape, nseq, backward)
 * bytes (it also holds each sequence's chunk offsets, which the call
 * derives from cu_seqlens on the device), the backward recomputes its
 * context (there is no saved-context pair), and offsets that do not rise
 * from 0 to T are found on the device: nothing is computed and
 * gdn_device_status() then returns GDN_ERR_SEQLENS. */
GDN_API size_t gdn_varlen_workspace(const gdn_shape* shape, int nseq, int backward);
GDN_API size_t kda_varlen_workspace(const gdn_shape* shape, int nseq, int backward);
GDN_API size_t mamba2_varlen_workspace(const gdn_shape* shape, int nseq, int backward);
GDN_API int gdn_fwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq, const void* q,
                           const void* k, const void* v, const float* g, const float* beta,
                           const float* h0, void* o, float* ht, void* ws, size_t ws_bytes,
                           void* stream);
GDN_API int gdn_bwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq, const void* q,
                           const void* k, const void* v, const float* g, const float* beta,
                           const float* h0, const void* do_, const float* dht, void* dq,
                           void* dk, void* dv, float* dg, float* dbeta, float* dh0, void* ws,
                           size_t ws_bytes, void* stream);
GDN_API int kda_fwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq, const void* q,
                           const void* k, const void* v, const void* g, const float* beta,
                           const float* h0, void* o, float* ht, void* ws, size_t ws_bytes,
                           void* stream);
GDN_API int kda_bwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq, const void* q,
                           const void* k, const void* v, const void* g, const float* beta,
                           const float* h0, const void* do_, const float* dht, void* dq,
                           void* dk, void* dv, void* dg, float* dbeta, float* dh0, void* ws,
                           size_t ws_bytes, void* stream);
GDN_API int mamba2_fwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq,
                              const void* q, const void* k, const void* v, const float* g,
                              const float* beta, const float* h0, void* o, float* ht, void* ws,
                              size_t ws_bytes, void* stream);
GDN_API int mamba2_bwd_varlen(const gdn_shape* shape, const int* cu_seqlens, int nseq,
                              const void* q, const void* k, const void* v, const float* g,
                              const float* beta, const float* h0, const void* do_,
                              const float* dht, void* dq, void* dk, void* dv, float* dg,
                              float* dbeta, float* dh0, void* ws, size_t ws_bytes, void* stream);

/* Decode: the forward recurrence run token by token, for a few tokens per
 * sequence (T = 1 in single-token generation).  Same arguments, layout and
 * results as *_fwd (o and the final state), with no workspace: each (b, h)
 * state is read once from h0 and written once to ht, and kept in registers
 * in between.  ht may equal h0 (the state is updated in place); h0 NULL is the
 * zero state; ht NULL skips the final state.  shape->chunk is not used but
 * must be a valid value.  Any dk, dv <= 128 and either dtype.  Its cost is
 * the state traffic, 2 x 4 dk dv bytes per (b, h) per call, plus the tokens'
 * own bytes; for long sequences *_fwd is the right call.  Errors as for
 * *_fwd (there is no GDN_ERR_WORKSPACE). */
GDN_API int gdn_decode(const gdn_shape* shape, const void* q, const void* k, const void* v,
                       const float* g, const float* beta, const float* h0, void* o, float* ht,
                       void* stream);
GDN_API int kda_decode(const gdn_shape* shape, const void* q, const void* k, const void* v,
                       const void* g, const float* beta, const float* h0, void* o, float* ht,
                       void* stream);

/* The mixer's fused neighbours (Primus hybrid-LLM pretraining blog, section
 * "Recipe", table 4: the "FLA fusions" row fuses the short convolution and
 * the gated norm around each mixer; the same table's normalisation epsilon
 * is 1e-6).  Both are elementwise along the tokens and bound by memory
 * traffic; each reads its inputs once and writes its outputs once.
 *
 * Short convolution, per channel c of x [B, T, H*D] (row-major, channel
 * fastest) with weights w [H*D, W] (fp32, row-major):
 *   s[t, c] = sum_{i<W} w[c, i] * x[t - W + 1 + i, c]   (x = 0 before the
 *             start of the token's sequence),
 *   y = s * sigmoid(s) (SiLU), and with l2norm != 0 each token's D values of
 *   a head are scaled:  z[t, h, :] = scale * y / sqrt(sum(y^2) + eps),
 *   else z = y.  The q and k projections take l2norm = 1 (q and k of the
 *   mixer), v takes l2norm = 0.
 * The backward recomputes s from x (nothing is saved) and writes dx (same
 * layout and dtype as x) and dw [H*D, W] (fp32, overwritten, summed over all
 * tokens in a fixed order: bit-for-bit reproducible) from dz.  It needs
 * gdn_short_conv_bwd_workspace(shape) bytes of device workspace.
 *
 * shape: D in {32, 64, 128}; W in [1, 4]; dtype GDN_F32 or GDN_BF16 (x, z,
 * dz, dx); B, T, H >= 0 with B*T <= 2^30 and H <= 65535 (an empty problem
 * launches nothing).  Packed
 * sequences: cu_seqlens non-NULL, B = 1, T the total token count and
 * cu_seqlens a DEVICE array of nseq + 1 int32 offsets as for the *_varlen
 * mixer calls; the convolution restarts at every sequence start.  Offsets
 * that do not rise from 0 to T give unspecified outputs (every access stays
 * inside the arrays) and gdn_device_status() returns GDN_ERR_SEQLENS.  With
 * cu_seqlens NULL, nseq is ignored and each of the B rows is one sequence.
 * Every token tensor must be 16-byte aligned (GDN_ERR_ALIGN).  Errors:
 * GDN_ERR_ARG (NULL pointer, eps < 0), GDN_ERR_SHAPE, GDN_ERR_DTYPE,
 * GDN_ERR_ALIGN, GDN_ERR_WORKSPACE, GDN_ERR_CUDA.  All pointers are device
 * pointers owned by the caller; the calls are asynchronous on `stream`. */
typedef struct {
  int B, T, H, D, W;
  int dtype;
} gdn_conv_shape;

GDN_API int gdn_short_conv_fwd(const gdn_conv_shape* shape, const void* x, const float* w,
                               void* z, int l2norm, float scale, float eps,
                               const int* cu_seqlens, int nseq, void* stream);
GDN_API size_t gdn_short_conv_bwd_workspace(const gdn_conv_shape* shape);
GDN_API int gdn_short_conv_bwd(const gdn_conv_shape* shape, const void* x, const float* w,
                               const void* dz, void* dx, float* dw, int l2norm, float scale,
                               float eps, const int* cu_seqlens, int nseq, void* ws,
                               size_t ws_bytes, void* stream);

/* Gated RMS norm of the mixer output, per row of D values (a row is one
 * token of one head: o and gate [rows, D], e.g. [B, T, H, dv] with rows =
 * B*T*H), with weight [D] (fp32) shared by all rows:
 *   out = o / sqrt(mean(o^2) + eps) * weight * gate * sigmoid(gate).
 * The backward writes do_ and dgate (layout and dtype of o) and dweight [D]
 * (fp32, overwritten, reproducible sum) from dout; it needs
 * gdn_gated_rmsnorm_bwd_workspace(shape) bytes of device workspace.  D in
 * {32, 64, 128}; rows >= 0; dtype GDN_F32 or GDN_BF16; errors and alignment
 * as for the short convolution. */
typedef struct {
  long long rows;
  int D;
  int dtype;
} gdn_norm_shape;

GDN_API int gdn_gated_rmsnorm_fwd(const gdn_norm_shape* shape, const void* o, const void* gate,
                                  const float* weight, void* out, float eps, void* stream);
GDN_API size_t gdn_gated_rmsnorm_bwd_workspace(const gdn_norm_shape* shape);
GDN_API int gdn_gated_rmsnorm_bwd(const gdn_norm_shape* shape, const void* o, const void* gate,
                                  const float* weight, const void* dout, void* do_, void* dgate,
                                  float* dweight, float eps, void* ws, size_t ws_bytes,
                                  void* stream);

/* Human-readable name of a gdn_status value. */
GDN_API const char* gdn_status_str(int status);

/* cudaError_t of the most recent GDN_ERR_CUDA on the calling thread. */
GDN_API int gdn_last_cuda_error(void);

/* Reads and clears the device status word of the current device: GDN_OK,
 * GDN_ERR_DEVICE_TIMEOUT or GDN_ERR_SEQLENS.  Synchronises the current
 * device.  Returns GDN_ERR_CUDA if the read itself fails. */
GDN_API int gdn_device_status(void);

/* Exercises the device-side timeout path.  Launches one CTA on `stream` that
 * sets up an mbarrier and tensor memory as the scan kernels do, then waits on
 * the barrier for at most max_tries bounded polls (each suspends the waiting
 * threads for at most about 20 us) while nothing can complete it: no thread
 * arrives and no copy or tensor-core operation is in flight.  The wait runs
 * out, and the CTA takes the scan kernels' timeout branch: it records
 * GDN_ERR_DEVICE_TIMEOUT in the device status word, frees its tensor memory
 * and returns.  A following gdn_device_status() returns
 * GDN_ERR_DEVICE_TIMEOUT (and clears it); the context stays usable.
 * max_tries must be in [1, 1000] (GDN_ERR_ARG otherwise). */
GDN_API int gdn_wait_selftest(int max_tries, void* stream);

/* 1 if the tensor-core kernels would run for this shape, else 0 (GDN / KDA).
 * For KDA this is the kernel family of the shape; a sequence whose gates
 * decay too fast for it inside some chunk is still computed by the CUDA-core
 * kernels (see "Kernel selection" above). */
GDN_API int gdn_uses_tensor_cores(const gdn_shape* shape);
GDN_API int kda_uses_tensor_cores(const gdn_shape* shape);

/* GDN backward for callers that cannot allocate device memory (an allocator
 * callback that must not re-enter the allocator, a framework thread that only
 * receives tensors, a path that forbids allocation after start-up).  The
 * paper has no counterpart: this is a library convenience.  It is gdn_bwd
 * with the workspace taken from a fixed 32 MiB device array built into the
 * library, which every GPU that loads the library holds until the process
 * exits.  Arguments and results are those of gdn_bwd without ws/ws_bytes.
 * Shapes whose gdn_bwd_workspace() exceeds 32 MiB return GDN_ERR_WORKSPACE
 * and launch nothing.  All calls share the array: calls whose GPU work
 * overlaps (other streams, unordered host threads) race and give wrong
 * results.  The first call on each device looks up the array's address
 * (cudaGetSymbolAddress) and keeps it until the process exits; make that call
 * before any stream capture, and do not call cudaDeviceReset after it (the
 * kept address would be stale).  A failure of that set-up returns
 * GDN_ERR_CUDA, with the CUDA error in gdn_last_cuda_error(). */
GDN_API int gdn_bwd_noalloc(const gdn_shape* shape, const void* q, const void* k, const void* v,
                            const float* g, const float* beta, const float* h0,
                            const void* do_, const float* dht, void* dq, void* dk, void* dv,
                            float* dg, float* dbeta, float* dh0, void* stream);

/* Per-kernel timing without a profiler (calling thread only).
 * gdn_profile_begin(cap) starts recording: every kernel the library launches
 * from this thread is bracketed by a pair of CUDA events recorded on the
 * launch stream, for the first `cap` launches (the library creates the events
 * once and keeps them; it allocates no device memory).  gdn_profile_end()
 * stops recording and returns the number of launches seen since begin (also
 * those beyond cap).  gdn_profile_read() waits for the recorded events and
 * writes, for each recorded launch in order, its kernel id and its duration
 * in ms; it returns the number written (<= max).  gdn_kernel_name() names a
 * kernel id.  Returns GDN_ERR_CUDA if an event call fails. */
GDN_API int gdn_profile_begin(int cap);
GDN_API int gdn_profile_end(void);
GDN_API int gdn_profile_read(int* kernel_ids, float* ms, int max);
GDN_API const char* gdn_kernel_name(int kernel_id);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H_ */
