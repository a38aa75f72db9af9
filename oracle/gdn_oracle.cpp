// Test infrastructure only: the fp64 CPU oracle for the gated delta rule.
//
// Nothing in the library or its product path may call this file.  It is
// built (by the package's build step) so that the tests, the smoke check and
// the benchmark's CPU baseline can compare the CUDA kernels against it.  It
// shares no code, header or table with the CUDA sources.
//
// What it computes.  The token mixers named on the Primus hybrid-LLM
// pretraining blog (MI355X), section "How hybrid models are defined in
// Primus": Gated DeltaNet (GDN) adds the delta rule (the memory update
// rewrites the value stored under the current key instead of only adding to
// it) to a state with one scalar forget gate per head; Kimi Delta Attention
// (KDA) refines that gate to one value per key dimension.  Written out per
// (batch b, head h) over tokens t = 0..T-1, with the state kept as
// H = S^T (dk x dv, row d = key dimension):
//
//   P      = a_t * H                 GDN: a_t = exp(g_t) (scalar)
//            diag(a_t) * H           KDA: a_t[d] = exp(g_t[d])
//   vpred  = P^T k_t                 (dv)
//   u      = beta_t (v_t - vpred)    (dv)
//   H      = P + k_t u^T
//   o_t    = H^T q_t
//
// which is S_t = a_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T with
// S = H^T and o_t = S_t q_t; for KDA the decay is applied before the erase
// term.  The same blog describes Mamba2, on the same mixer list, as the
// scalar-gated state that GDN extends with the delta rule: its state only
// accumulates.  That mixer is this loop without the delta rule's prediction,
// vpred = 0, so that H = a_t H + beta_t k_t v_t^T (beta_t the write strength,
// k/v/q the state-space input, input projection and read-out); the "no delta"
// flag selects it, with either gate form.  The backward pass is plain reverse-mode differentiation of this loop
// (every H_t is kept, so nothing is recomputed).  All arithmetic is fp64 and
// follows the loop token by token: no chunking, no blocking, no reordering.
//
// Layout: token tensors [B,T,H,D] row-major (D contiguous); g is [B,T,H] for
// GDN and [B,T,H,dk] for KDA; beta is [B,T,H]; states are [B,H,dk,dv].
// Independent (b,h) sequences are spread over std::threads.

#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <new>
#include <thread>
#include <vector>
#include <atomic>

namespace {

struct Dims {
  int B, T, H, dk, dv, kda, no_delta;
  size_t tok(int b, int t, int h, int D) const {
    return (((size_t)b * T + t) * H + h) * (size_t)D;
  }
  size_t gate(int b, int t, int h) const {
    return kda ? tok(b, t, h, dk) : ((size_t)b * T + t) * H + h;
  }
  size_t state(int b, int h) const {
    return ((size_t)b * H + h) * (size_t)dk * dv;
  }
};

// Runs fn(b, h) for every sequence on up to nthreads threads.
template <class F>
void for_each_sequence(const Dims& d, int nthreads, F fn) {
  const int n = d.B * d.H;
  if (nthreads <= 0) {
    nthreads = (int)std::thread::hardware_concurrency();
    if (nthreads <= 0) nthreads = 1;
  }
  if (nthreads > n) nthreads = n;
  std::atomic<int> next(0);
  auto worker = [&]() {
    for (;;) {
      int i = next.fetch_add(1);
      if (i >= n) break;
      fn(i / d.H, i % d.H);
    }
  };
  std::vector<std::thread> pool;
  for (int i = 1; i < nthreads; ++i) pool.emplace_back(worker);
  worker();
  for (auto& th : pool) th.join();
}

// One forward token step.  Hprev -> Hnext (may alias: no), also returns
// vpred in vp.  P is written to Pbuf (dk*dv).
void token_step(const Dims& d, const double* Hprev, const double* kt,
                const double* vt, const double* gt, double bt, double* Pbuf,
                double* vp, double* Hnext) {
  const int dk = d.dk, dv = d.dv;
  for (int i = 0; i < dk; ++i) {
    const double a = std::exp(d.kda ? gt[i] : gt[0]);
    for (int j = 0; j < dv; ++j) Pbuf[(size_t)i * dv + j] = a * Hprev[(size_t)i * dv + j];
  }
  for (int j = 0; j < dv; ++j) vp[j] = 0.0;
  if (!d.no_delta)
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) vp[j] += Pbuf[(size_t)i * dv + j] * kt[i];
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) {
      const double u = bt * (vt[j] - vp[j]);
      Hnext[(size_t)i * dv + j] = Pbuf[(size_t)i * dv + j] + kt[i] * u;
    }
}

}  // namespace

extern "C" {

// mode: bit 0 = one gate per key dimension (KDA), bit 1 = no delta rule.
//
// Forward.  h0 may be NULL (zero initial state); ht may be NULL.
// Returns 0 on success, -1 on bad arguments.
int oracle_fwd(int mode, int B, int T, int H, int dk, int dv, const double* q,
               const double* k, const double* v, const double* g,
               const double* beta, const double* h0, double* o, double* ht,
               int nthreads) {
  if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
  if (B == 0 || H == 0) return 0;
  const Dims d{B, T, H, dk, dv, mode & 1, (mode >> 1) & 1};
  for_each_sequence(d, nthreads, [&](int b, int h) {
    std::vector<double> Hs((size_t)dk * dv, 0.0), Hn((size_t)dk * dv), P((size_t)dk * dv);
    std::vector<double> vp(dv);
    if (h0) std::memcpy(Hs.data(), h0 + d.state(b, h), sizeof(double) * dk * dv);
    for (int t = 0; t < T; ++t) {
      const double* kt = k + d.tok(b, t, h, dk);
      const double* vt = v + d.tok(b, t, h, dv);
      const double* qt = q + d.tok(b, t, h, dk);
      token_step(d, Hs.data(), kt, vt, g + d.gate(b, t, h), beta[((size_t)b * T + t) * H + h],
                 P.data(), vp.data(), Hn.data());
      Hs.swap(Hn);
      double* ot = o + d.tok(b, t, h, dv);
      for (int j = 0; j < dv; ++j) ot[j] = 0.0;
      for (int i = 0; i < dk; ++i)
        for (int j = 0; j < dv; ++j) ot[j] += Hs[(size_t)i * dv + j] * qt[i];
    }
    if (ht) std::memcpy(ht + d.state(b, h), Hs.data(), sizeof(double) * dk * dv);
  });
  return 0;
}

// Backward (reverse mode of oracle_fwd).  h0 and dht may be NULL (zero);
// dh0 may be NULL (not wanted).  Keeps every H_t of one sequence in memory:
// T*dk*dv doubles per worker thread; refuses (-2) above 2^26 doubles.
int oracle_bwd(int mode, int B, int T, int H, int dk, int dv, const double* q,
               const double* k, const double* v, const double* g,
               const double* beta, const double* h0, const double* dout,
               const double* dht, double* dq, double* dk_, double* dv_,
               double* dg, double* dbeta, double* dh0, int nthreads) {
  if (B < 0 || T < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
  if ((double)(T + 1) * dk * dv > (double)(1u << 26)) return -2;
  if (B == 0 || H == 0) return 0;
  const Dims d{B, T, H, dk, dv, mode & 1, (mode >> 1) & 1};
  const size_t S = (size_t)dk * dv;
  for_each_sequence(d, nthreads, [&](int b, int h) {
    // Hall[t] = state after token t-1 (Hall[0] = h0); Hall[T] = final.
    std::vector<double> Hall((size_t)(T + 1) * S, 0.0);
    std::vector<double> P(S), vp(dv);
    if (h0) std::memcpy(Hall.data(), h0 + d.state(b, h), sizeof(double) * S);
    for (int t = 0; t < T; ++t)
      token_step(d, &Hall[(size_t)t * S], k + d.tok(b, t, h, dk), v + d.tok(b, t, h, dv),
                 g + d.gate(b, t, h), beta[((size_t)b * T + t) * H + h], P.data(), vp.data(),
                 &Hall[(size_t)(t + 1) * S]);

    std::vector<double> dH(S, 0.0), dP(S), du(dv), dvp(dv);
    if (dht) std::memcpy(dH.data(), dht + d.state(b, h), sizeof(double) * S);
    for (int t = T - 1; t >= 0; --t) {
      const double* qt = q + d.tok(b, t, h, dk);
      const double* kt = k + d.tok(b, t, h, dk);
      const double* vt = v + d.tok(b, t, h, dv);
      const double* gt = g + d.gate(b, t, h);
      const double bt = beta[((size_t)b * T + t) * H + h];
      const double* dot = dout + d.tok(b, t, h, dv);
      const double* Hprev = &Hall[(size_t)t * S];
      const double* Hcur = &Hall[(size_t)(t + 1) * S];
      double* dqt = dq + d.tok(b, t, h, dk);
      double* dkt = dk_ + d.tok(b, t, h, dk);
      double* dvt = dv_ + d.tok(b, t, h, dv);
      // recompute P_t and vpred_t
      for (int i = 0; i < dk; ++i) {
        const double a = std::exp(d.kda ? gt[i] : gt[0]);
        for (int j = 0; j < dv; ++j) P[(size_t)i * dv + j] = a * Hprev[(size_t)i * dv + j];
      }
      for (int j = 0; j < dv; ++j) vp[j] = 0.0;
      if (!d.no_delta)
        for (int i = 0; i < dk; ++i)
          for (int j = 0; j < dv; ++j) vp[j] += P[(size_t)i * dv + j] * kt[i];
      // o_t = H_t^T q_t
      for (int i = 0; i < dk; ++i) {
        double s = 0.0;
        for (int j = 0; j < dv; ++j) {
          s += Hcur[(size_t)i * dv + j] * dot[j];
          dH[(size_t)i * dv + j] += qt[i] * dot[j];
        }
        dqt[i] = s;
      }
      // H_t = P + k u^T
      for (int j = 0; j < dv; ++j) du[j] = 0.0;
      for (int i = 0; i < dk; ++i) {
        double s = 0.0;
        for (int j = 0; j < dv; ++j) {
          const double u = bt * (vt[j] - vp[j]);
          s += dH[(size_t)i * dv + j] * u;
          du[j] += dH[(size_t)i * dv + j] * kt[i];
        }
        dkt[i] = s;
      }
      // u = beta (v - vpred)
      double db = 0.0;
      for (int j = 0; j < dv; ++j) {
        dvt[j] = bt * du[j];
        db += du[j] * (vt[j] - vp[j]);
        dvp[j] = d.no_delta ? 0.0 : -bt * du[j];  // without the delta rule vpred is not formed
      }
      dbeta[((size_t)b * T + t) * H + h] = db;
      // vpred = P^T k ;  dP = dH + k dvp^T
      for (int i = 0; i < dk; ++i) {
        double s = 0.0;
        for (int j = 0; j < dv; ++j) {
          dP[(size_t)i * dv + j] = dH[(size_t)i * dv + j] + kt[i] * dvp[j];
          s += P[(size_t)i * dv + j] * dvp[j];
        }
        dkt[i] += s;
      }
      // P = a H_{t-1}
      if (d.kda) {
        double* dgt = dg + d.tok(b, t, h, dk);
        for (int i = 0; i < dk; ++i) {
          const double a = std::exp(gt[i]);
          double s = 0.0;
          for (int j = 0; j < dv; ++j) {
            s += dP[(size_t)i * dv + j] * P[(size_t)i * dv + j];
            dH[(size_t)i * dv + j] = a * dP[(size_t)i * dv + j];
          }
          dgt[i] = s;
        }
      } else {
        const double a = std::exp(gt[0]);
        double s = 0.0;
        for (size_t e = 0; e < S; ++e) {
          s += dP[e] * P[e];
          dH[e] = a * dP[e];
        }
        dg[((size_t)b * T + t) * H + h] = s;
      }
    }
    if (dh0) std::memcpy(dh0 + d.state(b, h), dH.data(), sizeof(double) * S);
  });
  return 0;
}

}  // extern "C"
