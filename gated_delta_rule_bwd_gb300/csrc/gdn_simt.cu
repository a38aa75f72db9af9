// CUDA-core (fp32 FFMA) chunkwise kernels for the GDN / KDA mixer.
//
// These run every shape the tensor-core kernels do not take: fp32 inputs
// (where bf16 tensor-core products cannot reach fp32 accuracy), head
// dimensions other than 128 and chunk sizes other than 64.  All arithmetic is
// fp32; inputs may be fp32 or bf16.
//
// Chunkwise form (per sequence, chunk of n <= C tokens, state H_in dk x dv;
// gamma = within-chunk cumulative sum of the log gate, per key dimension for
// KDA; Gam[r,j] = exp(gamma_r - gamma_j) for j <= r, elementwise per key
// dimension for KDA):
//   A = strict_lower(beta_r sum_d k_rd k_jd Gam[r,j,d])     (decayed K K^T)
//   R = V - (K o E) H_in,  E = exp(gamma)
//   U = (I + A)^-1 diag(beta) R                            (WY / UT transform)
//   O = (Q o E) H_in + lower_incl(sum_d q_rd k_jd Gam[r,j,d]) U
//   H_out = diag(exp(gamma_last)) H_in + (K o exp(gamma_last - gamma))^T U
// The forward triangular solve is a forward substitution; the backward pass
// walks the chunks in reverse, recomputing A, P, R and U from the stored
// chunk-boundary states, and uses the transposed solve (back substitution).
//
// Parallel layout: one CTA per (sequence, slice of dv columns).  Every term
// of the forward pass and of the state-gradient recurrence separates over dv
// columns; the gradients that sum over dv (dq, dk, dg, dbeta) are written as
// per-slice partials and summed in a fixed order by a reduction kernel, so
// results are deterministic.  Zero-filled tail rows (k = q = v = 0, g = 0,
// beta = 0) contribute nothing, so ragged tails need no special case.

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T> __device__ __forceinline__ float ldf(const T* p);
template <> __device__ __forceinline__ float ldf<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void stf(T* p, float x);
template <> __device__ __forceinline__ void stf<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

struct SimtArgs {
  Problem p;
  int dvs;        // dv columns per CTA
  int nsplit;     // CTAs per sequence along dv
  float* states;  // [B*H][N][dk][dv] chunk-entry states (bwd) or nullptr
  float* part;    // partial sums of the backward pass
  const int* only;  // if set, the kernels run only the sequences bh with only[bh] != 0
};

__device__ __forceinline__ size_t tok(const Problem& p, int b, int t, int h, int D) {
  return (((size_t)b * p.T + t) * p.H + h) * (size_t)D;
}

// Shared-memory carve-out, identical in host and device code.
struct FwdSmem {
  int Hs, Ks, Qs, Rs, Us, As, Ps, gm, bt, E, F, total;
};
__host__ __device__ inline FwdSmem fwd_smem(int dk, int dvs, int C, bool kda) {
  const int lk = dk + 1, lc = C + 1, lg = kda ? lk : 1;
  FwdSmem s;
  int o = 0;
  s.Hs = o; o += dk * dvs;
  s.Ks = o; o += C * lk;
  s.Qs = o; o += C * lk;
  s.Rs = o; o += C * dvs;
  s.Us = o; o += C * dvs;
  s.As = o; o += C * lc;
  s.Ps = o; o += C * lc;
  s.gm = o; o += C * lg;
  s.bt = o; o += C;
  s.E = o; o += C;
  s.F = o; o += C;
  s.total = o;
  return s;
}

struct BwdSmem {
  int Hs, dHs, Ks, Qs, gm, bt, E, F, rs, Rs, Os, Us, Zs, Ms, Ps, Ds, last, total;
};
__host__ __device__ inline BwdSmem bwd_smem(int dk, int dvs, int C, bool kda) {
  const int lk = dk + 1, lc = C + 1, lg = kda ? lk : 1;
  BwdSmem s;
  int o = 0;
  s.Hs = o; o += dk * dvs;
  s.dHs = o; o += dk * dvs;
  s.Ks = o; o += C * lk;
  s.Qs = o; o += C * lk;
  s.gm = o; o += C * lg;
  s.bt = o; o += C;
  s.E = o; o += C;
  s.F = o; o += C;
  s.rs = o; o += C;
  s.Rs = o; o += C * dvs;
  s.Os = o; o += C * dvs;
  s.Us = o; o += C * dvs;
  s.Zs = o; o += C * dvs;
  s.Ms = o; o += C * lc;
  s.Ps = o; o += C * lc;
  s.Ds = o; o += C * lc;
  s.last = o; o += dk;
  s.total = o;
  return s;
}

// Group of G consecutive lanes per dv column for the triangular solves.
__device__ __forceinline__ int solve_group(int nv) {
  int G = 32;
  while (G > 1 && G * nv > kThreads) G >>= 1;
  return G;
}

// Y_r = s_r * (X_r - sum_{j<r} M[r][j] Y_j), r = 0..n-1, columns < nv.
// With s = beta and M = beta-free decayed K K^T this is U = (I+A)^-1 diag(beta) R.
__device__ void forward_subst(const float* M, int lm, const float* s, const float* X, float* Y,
                              int ld, int nv, int n) {
  const int G = solve_group(nv);
  const int col = threadIdx.x / G, sub = threadIdx.x % G;
  const bool act = col < nv;
  for (int r = 0; r < n; ++r) {
    float acc = 0.f;
    if (act)
      for (int j = sub; j < r; j += G) acc += M[r * lm + j] * Y[j * ld + col];
    for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (act && sub == 0) Y[r * ld + col] = s[r] * (X[r * ld + col] - acc);
    __syncwarp();
  }
}

// In place: Z_r = Z_r - sum_{j>r} s_j M[j][r] Z_j, r = n-1..0  ((I+A)^T Z = dU).
__device__ void backward_subst(const float* M, int lm, const float* s, float* Z, int ld, int nv,
                               int n) {
  const int G = solve_group(nv);
  const int col = threadIdx.x / G, sub = threadIdx.x % G;
  const bool act = col < nv;
  for (int r = n - 1; r >= 0; --r) {
    float acc = 0.f;
    if (act)
      for (int j = r + 1 + sub; j < n; j += G) acc += s[j] * M[j * lm + r] * Z[j * ld + col];
    for (int off = G >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (act && sub == 0) Z[r * ld + col] -= acc;
    __syncwarp();
  }
}

// Loads the chunk's K, Q (zero-filled past the tail), g and beta, then turns g
// into gamma (inclusive cumsum) and, for GDN, E = exp(gamma) and
// F = exp(gamma_last - gamma).
template <typename TIn, bool KDA>
__device__ void load_chunk_keys(const Problem& p, int b, int h, int t0, int n, float* Ks,
                                float* Qs, float* gm, float* bt, float* E, float* F) {
  const int dk = p.dk, C = p.C, lk = dk + 1;
  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  for (int i = threadIdx.x; i < C * dk; i += kThreads) {
    const int r = i / dk, d = i % dk;
    float kv = 0.f, qv = 0.f;
    if (r < n) {
      const size_t o = tok(p, b, t0 + r, h, dk) + d;
      kv = ldf(k + o);
      qv = ldf(q + o);
    }
    Ks[r * lk + d] = kv;
    Qs[r * lk + d] = qv;
  }
  if (KDA) {
    for (int i = threadIdx.x; i < C * dk; i += kThreads) {
      const int r = i / dk, d = i % dk;
      gm[r * lk + d] = r < n ? gate_load(p, tok(p, b, t0 + r, h, dk) + d) : 0.f;
    }
  } else {
    for (int r = threadIdx.x; r < C; r += kThreads)
      gm[r] = r < n ? p.g[((size_t)b * p.T + t0 + r) * p.H + h] : 0.f;
  }
  for (int r = threadIdx.x; r < C; r += kThreads)
    bt[r] = r < n ? p.beta[((size_t)b * p.T + t0 + r) * p.H + h] : 0.f;
  __syncthreads();
  if (KDA) {
    for (int d = threadIdx.x; d < dk; d += kThreads) {
      float s = 0.f;
      for (int r = 0; r < C; ++r) {
        s += gm[r * lk + d];
        gm[r * lk + d] = s;
      }
    }
  } else if (threadIdx.x == 0) {
    float s = 0.f;
    for (int r = 0; r < C; ++r) {
      s += gm[r];
      gm[r] = s;
    }
  }
  __syncthreads();
  if (!KDA) {
    for (int r = threadIdx.x; r < C; r += kThreads) {
      E[r] = expf(gm[r]);
      F[r] = expf(gm[C - 1] - gm[r]);
    }
  }
  __syncthreads();
}

// decayed products of rows r >= j: sum_d x_rd y_jd Gam[r,j,d]
template <bool KDA>
__device__ __forceinline__ float decayed_dot(const float* X, const float* Y, const float* gm,
                                             int r, int j, int dk) {
  const int lk = dk + 1;
  float s = 0.f;
  if (KDA) {
    for (int d = 0; d < dk; ++d)
      s += X[r * lk + d] * Y[j * lk + d] * expf(gm[r * lk + d] - gm[j * lk + d]);
  } else {
    for (int d = 0; d < dk; ++d) s += X[r * lk + d] * Y[j * lk + d];
    s *= expf(gm[r] - gm[j]);
  }
  return s;
}

// ---------------------------------------------------------------- forward
// grid (B*H, nsplit).  With a.states set, also records each chunk's entry
// state (the backward pass's recompute); with p.o == nullptr skips the output.
template <typename TIn, bool KDA>
__global__ void __launch_bounds__(kThreads) simt_fwd_kernel(SimtArgs a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int bh = blockIdx.x, sq = bh / p.H, h = bh % p.H;
  if (a.only && !a.only[bh]) return;
  const Seqs seqs = Seqs::of(p);
  int b, tb, len, nch;
  seqs.get(sq, b, tb, len, nch);
  const int dk = p.dk, C = p.C, dvs = a.dvs, lk = dk + 1, lc = C + 1;
  const int v0 = blockIdx.y * dvs, nv = min(dvs, p.dv - v0);
  const FwdSmem L = fwd_smem(dk, dvs, C, KDA);
  float *Hs = sm + L.Hs, *Ks = sm + L.Ks, *Qs = sm + L.Qs, *Rs = sm + L.Rs, *Us = sm + L.Us;
  float *As = sm + L.As, *Ps = sm + L.Ps, *gm = sm + L.gm, *bt = sm + L.bt, *E = sm + L.E,
        *F = sm + L.F;
  const TIn* v = static_cast<const TIn*>(p.v);
  TIn* o = static_cast<TIn*>(p.o);

  for (int i = threadIdx.x; i < dk * dvs; i += kThreads) {
    const int d = i / dvs, c = i % dvs;
    Hs[i] = (p.h0 && c < nv) ? p.h0[((size_t)bh * dk + d) * p.dv + v0 + c] : 0.f;
  }
  for (int ci = 0; ci < nch; ++ci) {
    const int t0 = tb + ci * C, n = min(C, len - ci * C);  // t0: token within batch row b
    __syncthreads();
    if (a.states) {
      float* st = a.states + seqs.rec(sq, h, ci) * dk * p.dv;
      for (int i = threadIdx.x; i < dk * nv; i += kThreads) {
        const int d = i / nv, c = i % nv;
        st[(size_t)d * p.dv + v0 + c] = Hs[d * dvs + c];
      }
    }
    for (int i = threadIdx.x; i < C * dvs; i += kThreads) {
      const int r = i / dvs, c = i % dvs;
      Rs[i] = (r < n && c < nv) ? ldf(v + tok(p, b, t0 + r, h, p.dv) + v0 + c) : 0.f;
    }
    load_chunk_keys<TIn, KDA>(p, b, h, t0, n, Ks, Qs, gm, bt, E, F);
    // decayed K K^T (strict lower, beta applied in the solve; zero without the
    // delta rule) and masked Q K^T
    for (int i = threadIdx.x; i < C * C; i += kThreads) {
      const int r = i / C, j = i % C;
      float av = 0.f, pv = 0.f;
      if (j <= r) {
        if (j < r && !p.no_delta) av = decayed_dot<KDA>(Ks, Ks, gm, r, j, dk);
        pv = decayed_dot<KDA>(Qs, Ks, gm, r, j, dk);
      }
      As[r * lc + j] = av;
      Ps[r * lc + j] = pv;
    }
    // R = V - (K o E) H_in  (R = V without the delta rule)
    for (int i = threadIdx.x; i < C * dvs && !p.no_delta; i += kThreads) {
      const int r = i / dvs, c = i % dvs;
      float s = 0.f;
      if (KDA) {
        for (int d = 0; d < dk; ++d) s += Ks[r * lk + d] * expf(gm[r * lk + d]) * Hs[d * dvs + c];
      } else {
        for (int d = 0; d < dk; ++d) s += Ks[r * lk + d] * Hs[d * dvs + c];
        s *= E[r];
      }
      Rs[i] -= s;
    }
    __syncthreads();
    forward_subst(As, lc, bt, Rs, Us, dvs, nv, C);
    __syncthreads();
    if (o) {
      for (int i = threadIdx.x; i < n * nv; i += kThreads) {
        const int r = i / nv, c = i % nv;
        float s = 0.f;
        if (KDA) {
          for (int d = 0; d < dk; ++d) s += Qs[r * lk + d] * expf(gm[r * lk + d]) * Hs[d * dvs + c];
        } else {
          for (int d = 0; d < dk; ++d) s += Qs[r * lk + d] * Hs[d * dvs + c];
          s *= E[r];
        }
        for (int j = 0; j <= r; ++j) s += Ps[r * lc + j] * Us[j * dvs + c];
        stf(o + tok(p, b, t0 + r, h, p.dv) + v0 + c, s);
      }
      __syncthreads();
    }
    // H_out = diag(exp(gamma_last)) H_in + (K o exp(gamma_last - gamma))^T U
    for (int i = threadIdx.x; i < dk * nv; i += kThreads) {
      const int d = i / nv, c = i % nv;
      float s = 0.f, ec;
      if (KDA) {
        const float gl = gm[(C - 1) * lk + d];
        for (int j = 0; j < C; ++j) s += Ks[j * lk + d] * expf(gl - gm[j * lk + d]) * Us[j * dvs + c];
        ec = expf(gl);
      } else {
        for (int j = 0; j < C; ++j) s += Ks[j * lk + d] * F[j] * Us[j * dvs + c];
        ec = E[C - 1];
      }
      Hs[d * dvs + c] = ec * Hs[d * dvs + c] + s;
    }
  }
  __syncthreads();
  if (p.ht) {
    for (int i = threadIdx.x; i < dk * nv; i += kThreads) {
      const int d = i / nv, c = i % nv;
      p.ht[((size_t)bh * dk + d) * p.dv + v0 + c] = Hs[d * dvs + c];
    }
  }
}

// ---------------------------------------------------------------- backward
// Partial-sum layout in the workspace (fp32): dq [S][B,T,H,dk], dk [S][B,T,H,dk],
// dgamma [S][B,T,H,GD] (GD = dk for KDA, 1 for GDN), dbeta [S][B,T,H].
struct PartLayout {
  size_t dq, dk, dgam, dbeta, total;  // offsets in floats
};
__host__ __device__ inline PartLayout part_layout(const Problem& p, int nsplit) {
  const size_t tokh = (size_t)p.B * p.T * p.H;
  const size_t GD = p.kda ? p.dk : 1;
  PartLayout L;
  L.dq = 0;
  L.dk = L.dq + nsplit * tokh * p.dk;
  L.dgam = L.dk + nsplit * tokh * p.dk;
  L.dbeta = L.dgam + nsplit * tokh * GD;
  L.total = L.dbeta + nsplit * tokh;
  return L;
}

template <typename TIn, bool KDA>
__global__ void __launch_bounds__(kThreads) simt_bwd_kernel(SimtArgs a) {
  extern __shared__ float sm[];
  const Problem& p = a.p;
  const int bh = blockIdx.x, sq = bh / p.H, h = bh % p.H, split = blockIdx.y;
  if (a.only && !a.only[bh]) return;
  const Seqs seqs = Seqs::of(p);
  int b, tb, len, nch;
  seqs.get(sq, b, tb, len, nch);
  const int dk = p.dk, C = p.C, dvs = a.dvs, lk = dk + 1, lc = C + 1;
  const int v0 = split * dvs, nv = min(dvs, p.dv - v0);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const BwdSmem L = bwd_smem(dk, dvs, C, KDA);
  float *Hs = sm + L.Hs, *dHs = sm + L.dHs, *Ks = sm + L.Ks, *Qs = sm + L.Qs, *gm = sm + L.gm;
  float *bt = sm + L.bt, *E = sm + L.E, *F = sm + L.F, *rs = sm + L.rs;
  float *Rs = sm + L.Rs, *Os = sm + L.Os, *Us = sm + L.Us, *Zs = sm + L.Zs;
  float *Ms = sm + L.Ms, *Ps = sm + L.Ps, *Ds = sm + L.Ds, *last = sm + L.last;
  const TIn* v = static_cast<const TIn*>(p.v);
  const TIn* dO = static_cast<const TIn*>(p.do_);
  TIn* dv = static_cast<TIn*>(p.dv_);
  const PartLayout PL = part_layout(p, a.nsplit);
  const size_t tokh = (size_t)p.B * p.T * p.H;
  const int GD = KDA ? dk : 1;
  float* pdq = a.part + PL.dq + (size_t)split * tokh * dk;
  float* pdk = a.part + PL.dk + (size_t)split * tokh * dk;
  float* pdg = a.part + PL.dgam + (size_t)split * tokh * GD;
  float* pdb = a.part + PL.dbeta + (size_t)split * tokh;

  for (int i = threadIdx.x; i < dk * dvs; i += kThreads) {
    const int d = i / dvs, c = i % dvs;
    dHs[i] = (p.dht && c < nv) ? p.dht[((size_t)bh * dk + d) * p.dv + v0 + c] : 0.f;
  }
  for (int ci = nch - 1; ci >= 0; --ci) {
    const int t0 = tb + ci * C, n = min(C, len - ci * C);  // t0: token within batch row b
    __syncthreads();
    {
      const float* st = a.states + seqs.rec(sq, h, ci) * dk * p.dv;
      for (int i = threadIdx.x; i < dk * dvs; i += kThreads) {
        const int d = i / dvs, c = i % dvs;
        Hs[i] = c < nv ? st[(size_t)d * p.dv + v0 + c] : 0.f;
      }
    }
    for (int i = threadIdx.x; i < C * dvs; i += kThreads) {
      const int r = i / dvs, c = i % dvs;
      const bool ok = r < n && c < nv;
      const size_t off = ok ? tok(p, b, t0 + r, h, p.dv) + v0 + c : 0;
      Rs[i] = ok ? ldf(v + off) : 0.f;
      Os[i] = ok ? ldf(dO + off) : 0.f;
    }
    load_chunk_keys<TIn, KDA>(p, b, h, t0, n, Ks, Qs, gm, bt, E, F);
    for (int i = threadIdx.x; i < C * C; i += kThreads) {
      const int r = i / C, j = i % C;
      float mv = 0.f, pv = 0.f;
      if (j <= r) {
        if (j < r && !p.no_delta) mv = decayed_dot<KDA>(Ks, Ks, gm, r, j, dk);
        pv = decayed_dot<KDA>(Qs, Ks, gm, r, j, dk);
      }
      Ms[r * lc + j] = mv;
      Ps[r * lc + j] = pv;
    }
    for (int i = threadIdx.x; i < C * dvs && !p.no_delta; i += kThreads) {
      const int r = i / dvs, c = i % dvs;
      float s = 0.f;
      if (KDA) {
        for (int d = 0; d < dk; ++d) s += Ks[r * lk + d] * expf(gm[r * lk + d]) * Hs[d * dvs + c];
      } else {
        for (int d = 0; d < dk; ++d) s += Ks[r * lk + d] * Hs[d * dvs + c];
        s *= E[r];
      }
      Rs[i] -= s;
    }
    __syncthreads();
    forward_subst(Ms, lc, bt, Rs, Us, dvs, nv, C);
    __syncthreads();
    // dU = (K o F) dH_out + P^T dO
    for (int i = threadIdx.x; i < C * dvs; i += kThreads) {
      const int r = i / dvs, c = i % dvs;
      float s = 0.f;
      if (KDA) {
        const float* gl = gm + (C - 1) * lk;
        for (int d = 0; d < dk; ++d)
          s += Ks[r * lk + d] * expf(gl[d] - gm[r * lk + d]) * dHs[d * dvs + c];
      } else {
        for (int d = 0; d < dk; ++d) s += Ks[r * lk + d] * dHs[d * dvs + c];
        s *= F[r];
      }
      for (int j = r; j < C; ++j) s += Ps[j * lc + r] * Os[j * dvs + c];
      Zs[i] = s;
    }
    __syncthreads();
    backward_subst(Ms, lc, bt, Zs, dvs, nv, C);  // Zs = dZ
    __syncthreads();
    // C x C stage: dP (incl. lower), dA (strict lower); beta gradient parts
    for (int i = threadIdx.x; i < C * C; i += kThreads) {
      const int r = i / C, j = i % C;
      float dp = 0.f, da = 0.f;
      if (j <= r) {
        for (int c = 0; c < nv; ++c) dp += Os[r * dvs + c] * Us[j * dvs + c];
        if (j < r && !p.no_delta) {
          for (int c = 0; c < nv; ++c) da -= Zs[r * dvs + c] * Us[j * dvs + c];
        }
      }
      Ps[r * lc + j] = dp;
      Ds[r * lc + j] = da;
    }
    __syncthreads();
    for (int r = threadIdx.x; r < C; r += kThreads) {
      float s = 0.f;
      for (int c = 0; c < nv; ++c) s += Zs[r * dvs + c] * Rs[r * dvs + c];
      for (int j = 0; j < r; ++j) s += Ds[r * lc + j] * Ms[r * lc + j];
      rs[r] = s;  // dbeta partial
    }
    __syncthreads();
    for (int i = threadIdx.x; i < C * C; i += kThreads) {
      const int r = i / C, j = i % C;
      Ds[r * lc + j] *= bt[r];  // dA~ = beta_r dA_rj
    }
    for (int i = threadIdx.x; i < C * dvs; i += kThreads) Zs[i] *= bt[i / dvs];  // dR
    // gradient of gamma at the last row from H_out's decay factors
    for (int d = threadIdx.x; d < dk; d += kThreads) {
      float s1 = 0.f, s2 = 0.f;
      for (int c = 0; c < nv; ++c) s1 += dHs[d * dvs + c] * Hs[d * dvs + c];
      const float gl = KDA ? gm[(C - 1) * lk + d] : gm[C - 1];
      for (int j = 0; j < C; ++j) {
        float udh = 0.f;
        for (int c = 0; c < nv; ++c) udh += Us[j * dvs + c] * dHs[d * dvs + c];
        const float f = KDA ? expf(gl - gm[j * lk + d]) : F[j];
        s2 += Ks[j * lk + d] * f * udh;
      }
      last[d] = expf(gl) * s1 + s2;
    }
    __syncthreads();
    // per (row, key dim): dq, dk and dgamma partials
    for (int r = warp; r < n; r += kWarps) {
      float gsum = 0.f;
      for (int d = lane; d < dk; d += 32) {
        float dqe = 0.f, udh = 0.f, drh = 0.f;
        for (int c = 0; c < nv; ++c) {
          const float hdc = Hs[d * dvs + c];
          dqe += Os[r * dvs + c] * hdc;
          udh += Us[r * dvs + c] * dHs[d * dvs + c];
          drh += Zs[r * dvs + c] * hdc;
        }
        if (p.no_delta) drh = 0.f;  // R holds no state term
        float dqp = 0.f, dkp = 0.f, x = 0.f, y = 0.f;
        const float gr = KDA ? gm[r * lk + d] : gm[r];
        for (int j = 0; j <= r; ++j) {
          const float gj = KDA ? gm[j * lk + d] : gm[j];
          const float w = expf(gr - gj);
          dqp += Ps[r * lc + j] * Ks[j * lk + d] * w;
          x += Ds[r * lc + j] * Ks[j * lk + d] * w;
        }
        for (int j = r; j < C; ++j) {
          const float gj = KDA ? gm[j * lk + d] : gm[j];
          const float w = expf(gj - gr);
          dkp += Ps[j * lc + r] * Qs[j * lk + d] * w;
          y += Ds[j * lc + r] * Ks[j * lk + d] * w;
        }
        const float gl = KDA ? gm[(C - 1) * lk + d] : gm[C - 1];
        const float e = expf(gr), f = expf(gl - gr);
        const float qd = Qs[r * lk + d], kd = Ks[r * lk + d];
        const size_t off = tok(p, b, t0 + r, h, dk) + d;
        pdq[off] = e * dqe + dqp;
        pdk[off] = f * udh + dkp - e * drh + x + y;
        float dgam = qd * e * dqe + qd * dqp - kd * dkp + kd * x - kd * y - kd * e * drh -
                     kd * f * udh;
        if (r == n - 1) dgam += last[d];
        if (KDA) pdg[off] = dgam;
        else gsum += dgam;
      }
      if (!KDA) {
        for (int off = 16; off > 0; off >>= 1) gsum += __shfl_xor_sync(0xffffffffu, gsum, off);
        if (lane == 0) pdg[((size_t)b * p.T + t0 + r) * p.H + h] = gsum;
      }
      if (lane == 0) pdb[((size_t)b * p.T + t0 + r) * p.H + h] = rs[r];
    }
    // dv = dR
    for (int i = threadIdx.x; i < n * nv; i += kThreads) {
      const int r = i / nv, c = i % nv;
      stf(dv + tok(p, b, t0 + r, h, p.dv) + v0 + c, Zs[r * dvs + c]);
    }
    __syncthreads();
    // dH_in = diag(exp(gamma_last)) dH_out + (Q o E)^T dO - (K o E)^T dR
    // (without the delta rule R holds no state term: no dR part)
    const float kr = p.no_delta ? 0.f : 1.f;
    for (int i = threadIdx.x; i < dk * nv; i += kThreads) {
      const int d = i / nv, c = i % nv;
      float s = 0.f, ec;
      if (KDA) {
        for (int r = 0; r < C; ++r)
          s += expf(gm[r * lk + d]) *
               (Qs[r * lk + d] * Os[r * dvs + c] - kr * Ks[r * lk + d] * Zs[r * dvs + c]);
        ec = expf(gm[(C - 1) * lk + d]);
      } else {
        for (int r = 0; r < C; ++r)
          s += E[r] * (Qs[r * lk + d] * Os[r * dvs + c] - kr * Ks[r * lk + d] * Zs[r * dvs + c]);
        ec = E[C - 1];
      }
      dHs[d * dvs + c] = ec * dHs[d * dvs + c] + s;
    }
  }
  __syncthreads();
  if (p.dh0) {
    for (int i = threadIdx.x; i < dk * nv; i += kThreads) {
      const int d = i / nv, c = i % nv;
      p.dh0[((size_t)bh * dk + d) * p.dv + v0 + c] = dHs[d * dvs + c];
    }
  }
}

// Sums the per-slice partials in slice order and turns d(gamma) into d(g) by a
// reverse cumulative sum inside each chunk.  grid (B*H, N).
template <typename TIn, bool KDA>
__global__ void __launch_bounds__(kThreads) simt_bwd_reduce_kernel(SimtArgs a) {
  const Problem& p = a.p;
  const Seqs seqs = Seqs::of(p);
  int sq, h, ci, b, tb, len, nch;
  if (!seqs.chunk_of(blockIdx.x, p.nseq, sq, h, ci)) return;  // past the last packed chunk
  if (a.only && !a.only[sq * p.H + h]) return;
  seqs.get(sq, b, tb, len, nch);
  if (ci >= nch) return;
  const int dk = p.dk, t0 = tb + ci * p.C, n = min(p.C, len - ci * p.C);
  const PartLayout PL = part_layout(p, a.nsplit);
  const size_t tokh = (size_t)p.B * p.T * p.H;
  const int GD = KDA ? dk : 1;
  TIn* dq = static_cast<TIn*>(p.dq);
  TIn* dk_ = static_cast<TIn*>(p.dk_);
  for (int i = threadIdx.x; i < n * dk; i += kThreads) {
    const int r = i / dk, d = i % dk;
    const size_t off = tok(p, b, t0 + r, h, dk) + d;
    float sq = 0.f, sk = 0.f;
    for (int s = 0; s < a.nsplit; ++s) {
      sq += a.part[PL.dq + s * tokh * dk + off];
      sk += a.part[PL.dk + s * tokh * dk + off];
    }
    stf(dq + off, sq);
    stf(dk_ + off, sk);
  }
  for (int r = threadIdx.x; r < n; r += kThreads) {
    const size_t off = ((size_t)b * p.T + t0 + r) * p.H + h;
    float s = 0.f;
    for (int sp = 0; sp < a.nsplit; ++sp) s += a.part[PL.dbeta + sp * tokh + off];
    p.dbeta[off] = s;
  }
  for (int d = threadIdx.x; d < GD; d += kThreads) {
    float run = 0.f;
    for (int r = n - 1; r >= 0; --r) {
      const size_t off = KDA ? tok(p, b, t0 + r, h, dk) + d : ((size_t)b * p.T + t0 + r) * p.H + h;
      float s = 0.f;
      for (int sp = 0; sp < a.nsplit; ++sp) s += a.part[PL.dgam + sp * tokh * GD + off];
      run += s;
      dgate_store(p, off, run);
    }
  }
}

constexpr size_t kSmemLimit = 227 * 1024;

// dv columns per CTA: the widest slice (<= 32) whose shared memory fits.
int pick_dvs_fwd(const Problem& p) {
  for (int dvs : {32, 16, 8, 4, 2, 1})
    if ((size_t)fwd_smem(p.dk, dvs, p.C, p.kda).total * 4 <= kSmemLimit)
      return dvs < p.dv ? dvs : p.dv;
  return 1;
}
int pick_dvs_bwd(const Problem& p) {
  for (int dvs : {32, 16, 8, 4, 2, 1})
    if ((size_t)bwd_smem(p.dk, dvs, p.C, p.kda).total * 4 <= kSmemLimit)
      return dvs < p.dv ? dvs : p.dv;
  return 1;
}

size_t states_bytes(const Problem& p) {
  return align_up((size_t)max_chunks(p) * p.H * p.dk * p.dv * sizeof(float), 256);
}

template <typename TIn, bool KDA>
cudaError_t launch_fwd(const Problem& p, cudaStream_t s, float* states, bool want_out,
                       const int* only) {
  const int kid = want_out ? kSimtFwd : kSimtStates;
  SimtArgs a{};
  a.p = p;
  a.only = only;
  if (!want_out) a.p.o = nullptr, a.p.ht = nullptr;
  a.dvs = pick_dvs_fwd(p);
  a.nsplit = (p.dv + a.dvs - 1) / a.dvs;
  a.states = states;
  const size_t smem = (size_t)fwd_smem(p.dk, a.dvs, p.C, KDA).total * sizeof(float);
  auto kern = simt_fwd_kernel<TIn, KDA>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_before(s);
  kern<<<dim3(num_seqs(p) * p.H, a.nsplit), kThreads, smem, s>>>(a);
  prof_after(s, kid);
  return cudaGetLastError();
}

// With saved, the workspace holds the entry states that launch_fwd wrote
// alongside the output (a saved context), and the states pass is skipped.
template <typename TIn, bool KDA>
cudaError_t launch_bwd(const Problem& p, cudaStream_t s, bool saved, const int* only) {
  float* states = static_cast<float*>(p.ws);
  cudaError_t e;
  if (!saved && (e = launch_fwd<TIn, KDA>(p, s, states, false, only)) != cudaSuccess) return e;
  SimtArgs a{};
  a.p = p;
  a.only = only;
  a.dvs = pick_dvs_bwd(p);
  a.nsplit = (p.dv + a.dvs - 1) / a.dvs;
  a.states = states;
  a.part = reinterpret_cast<float*>(static_cast<char*>(p.ws) + states_bytes(p));
  const size_t smem = (size_t)bwd_smem(p.dk, a.dvs, p.C, KDA).total * sizeof(float);
  auto kern = simt_bwd_kernel<TIn, KDA>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prof_before(s);
  kern<<<dim3(num_seqs(p) * p.H, a.nsplit), kThreads, smem, s>>>(a);
  prof_after(s, kSimtBwd);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_before(s);
  simt_bwd_reduce_kernel<TIn, KDA><<<(unsigned)(max_chunks(p) * p.H), kThreads, 0, s>>>(a);
  prof_after(s, kSimtBwdReduce);
  return cudaGetLastError();
}

}  // namespace

size_t simt_bwd_workspace(const Problem& p) {
  const int dvs = pick_dvs_bwd(p);
  const int nsplit = (p.dv + dvs - 1) / dvs;
  return states_bytes(p) + align_up(part_layout(p, nsplit).total * sizeof(float), 256);
}

cudaError_t simt_fwd(const Problem& p, cudaStream_t s, bool save, const int* only) {
  float* st = save ? static_cast<float*>(p.ws) : nullptr;
  if (p.bf16) return p.kda ? launch_fwd<__nv_bfloat16, true>(p, s, st, true, only)
                           : launch_fwd<__nv_bfloat16, false>(p, s, st, true, only);
  return p.kda ? launch_fwd<float, true>(p, s, st, true, only)
               : launch_fwd<float, false>(p, s, st, true, only);
}

cudaError_t simt_bwd(const Problem& p, cudaStream_t s, bool saved, const int* only) {
  if (p.bf16)
    return p.kda ? launch_bwd<__nv_bfloat16, true>(p, s, saved, only)
                 : launch_bwd<__nv_bfloat16, false>(p, s, saved, only);
  return p.kda ? launch_bwd<float, true>(p, s, saved, only)
               : launch_bwd<float, false>(p, s, saved, only);
}

}  // namespace gdn
