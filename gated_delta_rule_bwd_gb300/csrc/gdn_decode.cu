// Token-recurrent forward for a few tokens per sequence (decode).
//
// The recurrence of the mixers (Primus hybrid-LLM pretraining blog, section
// "How hybrid models are defined in Primus"), one token at a time, per batch
// row b and head h, with the state H (dk x dv, fp32):
//   GDN:  P = exp(g_t) H          KDA:  P = diag(exp(g_t)) H
//   u = beta_t (v_t - P^T k_t),   H <- P + k_t u^T,   o_t = H^T q_t
// o_t = P^T q_t + (k_t . q_t) u, so one pass over H gives P^T k and P^T q.
//
// Every term separates over the value columns, so one warp owns 16 columns of
// one (b, h) state and keeps them in registers (two lanes per column, 64 rows
// each) for all T tokens: the state is read from HBM once and written once
// per call, and each token adds only its q, k, v, o, g and beta.  The token's
// k, its decay a = exp(g) per key row and the products a k, a q go through a
// per-warp shared-memory slice that every lane reads by broadcast:
// P^T k = H^T (a k), P^T q = H^T (a q), and H <- diag(a) H + k u^T.  This
// path is bound by the state traffic (2 x 4 dk dv bytes per (b, h) per call);
// long sequences belong to the chunkwise kernels.

#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kDecWarps = 2;  // warps per CTA
constexpr int kMaxD = 128;
constexpr int kCols = 16;     // state columns per warp
constexpr int kRows = 64;     // state rows per lane (two lanes per column)

template <typename T> __device__ __forceinline__ float dld(const T* p);
template <> __device__ __forceinline__ float dld<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float dld<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}
template <typename T> __device__ __forceinline__ void dst_(T* p, float x);
template <> __device__ __forceinline__ void dst_<float>(float* p, float x) { *p = x; }
template <> __device__ __forceinline__ void dst_<__nv_bfloat16>(__nv_bfloat16* p, float x) {
  *p = __float2bfloat16_rn(x);
}

// FULL: dk = dv = 128, known at compile time (no row or column guards, and
// constant strides).  Lane l of a warp holds column 16 s + (l % 16) of the
// state, rows 64 (l / 16) + [0, 64): two lanes share a column and join their
// partial sums with one shuffle.
template <typename TIn, bool KDA, bool FULL>
__global__ void __launch_bounds__(32 * kDecWarps) decode_kernel(Problem p) {
  // the token's k, decay a = exp(g) per key row (GDN: one value repeated),
  // a k and a q
  __shared__ __align__(16) float vec[kDecWarps][4][kMaxD];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int nsl = FULL ? kMaxD / kCols : (p.dv + kCols - 1) / kCols;
  const long gw = (long)blockIdx.x * kDecWarps + wi;
  if (gw >= (long)p.B * p.H * nsl) return;  // whole warps only: no later block-wide barrier
  const int bh = (int)(gw / nsl), sl = (int)(gw % nsl), b = bh / p.H, h = bh % p.H;
  const int dk = FULL ? kMaxD : p.dk, dv = FULL ? kMaxD : p.dv;
  const int c = sl * kCols + (lane & (kCols - 1)), r0 = (lane / kCols) * kRows;
  const bool act = c < dv;
  float* const kv = &vec[wi][0][0];
  float* const av = kv + kMaxD;
  float* const kav = kv + 2 * kMaxD;
  float* const qav = kv + 3 * kMaxD;
  const TIn* q = static_cast<const TIn*>(p.q);
  const TIn* k = static_cast<const TIn*>(p.k);
  const TIn* v = static_cast<const TIn*>(p.v);
  TIn* o = static_cast<TIn*>(p.o);

  float hc[kRows];  // rows r0 + [0, 64) of column c of the state
  const float* h0 = p.h0 ? p.h0 + (size_t)bh * dk * dv : nullptr;
#pragma unroll
  for (int i = 0; i < kRows; ++i)
    hc[i] = (r0 + i < dk && act && h0) ? h0[(size_t)(r0 + i) * dv + c] : 0.f;

  for (int t = 0; t < p.T; ++t) {
    const size_t tokh = ((size_t)b * p.T + t) * p.H + h;  // (b, t, h)
    __syncwarp();  // the previous token's vectors have been read
    float kq = 0.f;
    const float ag = KDA ? 0.f : expf(p.g[tokh]);
    for (int d = lane; d < kMaxD; d += 32) {  // zero past dk
      const bool in = d < dk;
      const float kd = in ? dld(k + tokh * dk + d) : 0.f, qd = in ? dld(q + tokh * dk + d) : 0.f;
      const float ad = !in ? 0.f : KDA ? expf(gate_load(p, tokh * dk + d)) : ag;
      kv[d] = kd;
      av[d] = ad;
      kav[d] = ad * kd;
      qav[d] = ad * qd;
      kq = fmaf(kd, qd, kq);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
    const float beta = p.beta[tokh];
    const float vc = act ? dld(v + tokh * dv + c) : 0.f;
    __syncwarp();
    // P^T k and P^T q over this lane's rows, through a k and a q (four
    // independent sums each; the vectors are read four at a time, by
    // broadcast within each half-warp), joined across the two lanes of the
    // column; then the update H <- diag(a) H + k u^T.
    float pk[4] = {0.f, 0.f, 0.f, 0.f}, pq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i4 = 0; i4 < kRows; i4 += 4) {
      if (FULL || r0 + i4 < dk) {
        const float4 k4 = *reinterpret_cast<const float4*>(kav + r0 + i4);
        const float4 q4 = *reinterpret_cast<const float4*>(qav + r0 + i4);
        const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, qq[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          pk[i] = fmaf(hc[i4 + i], kk[i], pk[i]);
          pq[i] = fmaf(hc[i4 + i], qq[i], pq[i]);
        }
      }
    }
    float ptk = (pk[0] + pk[1]) + (pk[2] + pk[3]), ptq = (pq[0] + pq[1]) + (pq[2] + pq[3]);
    ptk += __shfl_xor_sync(0xffffffffu, ptk, kCols);
    ptq += __shfl_xor_sync(0xffffffffu, ptq, kCols);
    const float u = beta * (vc - ptk);
    if (act && r0 == 0) dst_(o + tokh * dv + c, ptq + kq * u);
#pragma unroll
    for (int i4 = 0; i4 < kRows; i4 += 4) {
      if (FULL || r0 + i4 < dk) {
        const float4 k4 = *reinterpret_cast<const float4*>(kv + r0 + i4);
        const float4 a4 = *reinterpret_cast<const float4*>(av + r0 + i4);
        const float kk[4] = {k4.x, k4.y, k4.z, k4.w}, aa[4] = {a4.x, a4.y, a4.z, a4.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) hc[i4 + i] = fmaf(aa[i], hc[i4 + i], kk[i] * u);
      }
    }
  }
  if (p.ht && act) {
    float* ht = p.ht + (size_t)bh * dk * dv;
#pragma unroll
    for (int i = 0; i < kRows; ++i)
      if (r0 + i < dk) ht[(size_t)(r0 + i) * dv + c] = hc[i];
  }
}

template <typename TIn, bool KDA>
cudaError_t launch_decode(const Problem& p, cudaStream_t s) {
  const long warps = (long)p.B * p.H * ((p.dv + kCols - 1) / kCols);
  const unsigned grid = (unsigned)((warps + kDecWarps - 1) / kDecWarps);
  prof_before(s);
  if (p.dk == kMaxD && p.dv == kMaxD)
    decode_kernel<TIn, KDA, true><<<grid, 32 * kDecWarps, 0, s>>>(p);
  else
    decode_kernel<TIn, KDA, false><<<grid, 32 * kDecWarps, 0, s>>>(p);
  prof_after(s, kDecode);
  return cudaGetLastError();
}

}  // namespace

cudaError_t decode(const Problem& p, cudaStream_t s) {
  if (p.bf16) return p.kda ? launch_decode<__nv_bfloat16, true>(p, s)
                           : launch_decode<__nv_bfloat16, false>(p, s);
  return p.kda ? launch_decode<float, true>(p, s) : launch_decode<float, false>(p, s);
}

}  // namespace gdn
