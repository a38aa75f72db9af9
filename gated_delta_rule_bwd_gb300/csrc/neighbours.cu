// The mixer's fused neighbours: the short convolution in front of q, k and v
// (with the q/k L2 norm) and the gated RMS norm after o.
//
// The Primus hybrid-LLM pretraining blog (section "Recipe", table 4, the
// "FLA fusions" row) fuses both around every mixer, with the normalisation
// epsilon of the same table (1e-6):
//   short conv:  s_t = sum_i w_i x_{t-W+1+i} per channel (causal, zero before
//                the sequence start), y = SiLU(s); for q and k each head's D
//                values are then scaled to z = scale y / sqrt(|y|^2 + eps);
//   gated norm:  out = o / sqrt(mean(o^2) + eps) * weight * SiLU(gate) per
//                token and head over its D values.
//
// Both are bound by HBM: every element is read once and written once.  One
// warp owns one head's D channels of a token (D / 32 per lane), so the head's
// norms are warp shuffles and a token row is one coalesced access.
//
// Short conv: a warp walks a run of kRun consecutive tokens and keeps the
// previous W - 1 inputs of its channels in registers (the forward reads each
// row once plus a 3-row halo per run, which the neighbouring warp has just
// brought into L2).  The backward walks its run backwards, recomputing s from
// x (no saved activations), with the last three ds values of its channels in
// registers: dx_t = sum_i w_i ds_{t+W-1-i} needs ds of up to three later
// tokens, which come from a 3-token halo after the run.  dw is summed per
// warp in registers, per CTA in shared memory and over CTAs by a second
// kernel in a fixed order, so the result is bit-for-bit reproducible.
// Packed sequences split a run where a sequence ends; the windows restart
// from zeros there.
//
// Gated norm: a warp takes kNormRows rows at a time (all loads first, then
// the arithmetic); dweight is reduced like dw.

#include <algorithm>
#include <type_traits>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace gdn {
namespace {

__device__ int g_nb_status = 0;

constexpr int kNbWarps = 8;      // warps per CTA
constexpr int kRun = 32;         // tokens per warp run (short conv)
constexpr int kBatchFwd = 8;     // rows loaded ahead (short conv forward)
constexpr int kBatchBwd = 4;     // token steps loaded ahead (short conv backward)
constexpr int kNormRows = 4;     // rows per warp step (gated norm forward)
constexpr int kNormRowsBwd = 2;  // rows per warp step (gated norm backward)
constexpr int kMaxTaps = 4;      // widest convolution
constexpr int kConvGroupsTarget = 1024;  // CTAs of the backward conv (before the head split)
constexpr int kNormCtasMax = 512;

// ---------------------------------------------------------------- vector access
// One lane's EPL consecutive elements as one load: rows are prefetched in
// this packed form (bf16 pairs stay packed) and widened to fp32 on use.
template <typename T, int EPL> struct Raw;
template <> struct Raw<float, 4> { using type = float4; };
template <> struct Raw<float, 2> { using type = float2; };
template <> struct Raw<float, 1> { using type = float; };
template <> struct Raw<__nv_bfloat16, 4> { using type = uint2; };
template <> struct Raw<__nv_bfloat16, 2> { using type = uint32_t; };
template <> struct Raw<__nv_bfloat16, 1> { using type = unsigned short; };

template <typename T, int EPL>
__device__ __forceinline__ typename Raw<T, EPL>::type ldr(const T* __restrict__ p) {
  return *reinterpret_cast<const typename Raw<T, EPL>::type*>(p);
}

__device__ __forceinline__ float2 bf2(uint32_t u) {
  return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u));
}

template <typename T, int EPL>
__device__ __forceinline__ void widen(const typename Raw<T, EPL>::type& r, float (&v)[EPL]) {
  if constexpr (std::is_same<T, float>::value) {
    if constexpr (EPL == 4) {
      v[0] = r.x; v[1] = r.y; v[2] = r.z; v[3] = r.w;
    } else if constexpr (EPL == 2) {
      v[0] = r.x; v[1] = r.y;
    } else {
      v[0] = r;
    }
  } else {
    if constexpr (EPL == 4) {
      const float2 lo = bf2(r.x), hi = bf2(r.y);
      v[0] = lo.x; v[1] = lo.y; v[2] = hi.x; v[3] = hi.y;
    } else if constexpr (EPL == 2) {
      const float2 a = bf2(r);
      v[0] = a.x; v[1] = a.y;
    } else {
      v[0] = __uint_as_float((uint32_t)r << 16);
    }
  }
}

template <typename T, int EPL>
__device__ __forceinline__ void ldv(const T* __restrict__ p, float (&v)[EPL]) {
  widen<T, EPL>(ldr<T, EPL>(p), v);
}

template <typename T, int EPL>
__device__ __forceinline__ typename Raw<T, EPL>::type raw_zero() {
  typename Raw<T, EPL>::type r;
  memset(&r, 0, sizeof(r));
  return r;
}

template <typename T, int EPL>
__device__ __forceinline__ void stv(T* __restrict__ p, const float (&v)[EPL]) {
  if constexpr (std::is_same<T, float>::value) {
    if constexpr (EPL == 4) {
      *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
    } else if constexpr (EPL == 2) {
      *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    } else {
      *p = v[0];
    }
  } else {
    if constexpr (EPL == 4) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
      uint2 a;
      a.x = *reinterpret_cast<const uint32_t*>(&lo);
      a.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(p) = a;
    } else if constexpr (EPL == 2) {
      *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
    } else {
      *p = __float2bfloat16_rn(v[0]);
    }
  }
}

template <int EPL>
__device__ __forceinline__ void zero(float (&v)[EPL]) {
#pragma unroll
  for (int e = 0; e < EPL; ++e) v[e] = 0.f;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// Fast-math sigmoid: the quotient's error (a few ulp) is far below the bf16
// rounding of the outputs; for s < -87 it gives 0 (the exact value is below
// 1e-38).
__device__ __forceinline__ float sigmoid(float s) { return __fdividef(1.f, 1.f + __expf(-s)); }

// ---------------------------------------------------------------- sequence bounds
// The sequence [lo, hi) that holds flattened token t.  Fixed length: rows of
// T tokens.  Packed: the largest j with cu[j] <= t.  Both ends are clamped
// to [0, Ttot) around t, so that offsets that are not a valid partition
// (reported by the set-up check) still keep every access in bounds.
template <bool Packed>
__device__ __forceinline__ void seq_bounds(int t, int T, int Ttot, const int* __restrict__ cu,
                                           int nseq, int& lo, int& hi) {
  if constexpr (!Packed) {
    lo = t / T * T;
    hi = lo + T;
  } else {
    int a = 0, b = nseq;  // invariant: cu[a] <= t (when the offsets are valid)
    while (a < b) {
      const int m = (a + b + 1) >> 1;
      if (cu[m] <= t) a = m; else b = m - 1;
    }
    lo = cu[a];
    hi = a < nseq ? cu[a + 1] : Ttot;
  }
  lo = lo < 0 ? 0 : (lo > t ? t : lo);
  hi = hi > Ttot ? Ttot : (hi <= t ? t + 1 : hi);
}

// CTA 0 checks the packed offsets once: cu[0] = 0, cu[nseq] = Ttot and
// non-decreasing.  A bad partition sets GDN_ERR_SEQLENS in the status word.
__device__ void check_offsets(const int* __restrict__ cu, int nseq, int Ttot) {
  int bad = 0;
  if (threadIdx.x == 0) bad = cu[0] != 0 || cu[nseq] != Ttot;
  for (int j = threadIdx.x; j < nseq; j += blockDim.x) bad |= cu[j + 1] < cu[j];
  if (__syncthreads_or(bad) && threadIdx.x == 0) atomicExch(&g_nb_status, GDN_ERR_SEQLENS);
}

// Tap weights of lane channels, left-padded to kMaxTaps: wp[j] multiplies
// x_{t-3+j}, so a width W < 4 has zeros in its first 4 - W taps.
template <int EPL>
__device__ __forceinline__ void load_taps(const float* __restrict__ w, int W, int c0,
                                          float (&wp)[kMaxTaps][EPL]) {
#pragma unroll
  for (int j = 0; j < kMaxTaps; ++j)
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      const int i = j - (kMaxTaps - W);
      wp[j][e] = i >= 0 ? w[(long)(c0 + e) * W + i] : 0.f;
    }
}

struct ConvArgs {
  const void* x;
  const float* w;
  void* z;
  const void* dz;
  void* dx;
  float* part;  // backward: [gridDim.x][H*D*W] partial dw
  const int* cu;
  int nseq;
  int T;        // tokens per row (fixed length)
  int Ttot;     // all tokens (at most 2^30)
  int H, D, W;
  float scale, eps;
  int l2norm;
};

// ---------------------------------------------------------------- short conv forward
template <typename T, int EPL, bool Packed>
__global__ void __launch_bounds__(32 * kNbWarps, 2) short_conv_fwd_kernel(ConvArgs a) {
  if (Packed && blockIdx.x == 0 && blockIdx.y == 0) check_offsets(a.cu, a.nseq, a.Ttot);
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int h = blockIdx.y;
  const long CH = (long)a.H * a.D;
  const int c0 = h * a.D + lane * EPL;
  const T* __restrict__ x = static_cast<const T*>(a.x) + c0;
  T* __restrict__ z = static_cast<T*>(a.z) + c0;
  float wp[kMaxTaps][EPL];
  load_taps<EPL>(a.w, a.W, c0, wp);
  const int nruns = (a.Ttot + kRun - 1) / kRun;
#pragma unroll 1
  for (int r = blockIdx.x * kNbWarps + wi; r < nruns; r += gridDim.x * kNbWarps) {
    const int r1 = min((r + 1) * kRun, a.Ttot);
#pragma unroll 1
    for (int t0 = r * kRun; t0 < r1;) {
      int lo, hi;
      seq_bounds<Packed>(t0, a.T, a.Ttot, a.cu, a.nseq, lo, hi);
      const int t1 = min(r1, hi);
      float win[kMaxTaps - 1][EPL];  // x_{t-3}, x_{t-2}, x_{t-1}
#pragma unroll
      for (int j = 0; j < kMaxTaps - 1; ++j) {
        const int row = t0 - (kMaxTaps - 1) + j;
        if (row >= lo) ldv<T, EPL>(x + (long)row * CH, win[j]); else zero(win[j]);
      }
#pragma unroll 1
      for (int t = t0; t < t1; t += kBatchFwd) {
        typename Raw<T, EPL>::type xraw[kBatchFwd];
#pragma unroll
        for (int u = 0; u < kBatchFwd; ++u)
          if (t + u < t1) xraw[u] = ldr<T, EPL>(x + (long)(t + u) * CH);
#pragma unroll
        for (int u = 0; u < kBatchFwd; ++u) {
          if (t + u >= t1) break;
          float xr[EPL], y[EPL];
          widen<T, EPL>(xraw[u], xr);
          float ss = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            float s = wp[kMaxTaps - 1][e] * xr[e];
#pragma unroll
            for (int j = 0; j < kMaxTaps - 1; ++j) s = fmaf(wp[j][e], win[j][e], s);
            y[e] = s * sigmoid(s);
            ss = fmaf(y[e], y[e], ss);
          }
          if (a.l2norm) {
            const float r = a.scale * rsqrtf(warp_sum(ss) + a.eps);
#pragma unroll
            for (int e = 0; e < EPL; ++e) y[e] *= r;
          }
          stv<T, EPL>(z + (long)(t + u) * CH, y);
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            win[0][e] = win[1][e];
            win[1][e] = win[2][e];
            win[2][e] = xr[e];
          }
        }
      }
      t0 = t1;
    }
  }
}

// ---------------------------------------------------------------- short conv backward
template <typename T, int EPL, bool Packed>
__global__ void __launch_bounds__(32 * kNbWarps, 2) short_conv_bwd_kernel(ConvArgs a) {
  __shared__ float red[kNbWarps][kMaxTaps][128];
  if (Packed && blockIdx.x == 0 && blockIdx.y == 0) check_offsets(a.cu, a.nseq, a.Ttot);
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int h = blockIdx.y;
  const long CH = (long)a.H * a.D;
  const int c0 = h * a.D + lane * EPL;
  const T* __restrict__ x = static_cast<const T*>(a.x) + c0;
  const T* __restrict__ dz = static_cast<const T*>(a.dz) + c0;
  T* __restrict__ dx = static_cast<T*>(a.dx) + c0;
  float wp[kMaxTaps][EPL];
  load_taps<EPL>(a.w, a.W, c0, wp);
  float dwp[kMaxTaps][EPL];
#pragma unroll
  for (int j = 0; j < kMaxTaps; ++j) zero(dwp[j]);
  const int nruns = (a.Ttot + kRun - 1) / kRun;
#pragma unroll 1
  for (int r = blockIdx.x * kNbWarps + wi; r < nruns; r += gridDim.x * kNbWarps) {
    const int r1 = min((r + 1) * kRun, a.Ttot);
#pragma unroll 1
    for (int t0 = r * kRun; t0 < r1;) {
      int lo, hi;
      seq_bounds<Packed>(t0, a.T, a.Ttot, a.cu, a.nseq, lo, hi);
      const int t1 = min(r1, hi);             // own tokens [t0, t1)
      const int te = min(t1 + kMaxTaps - 1, hi);  // plus the halo [t1, te)
      typename Raw<T, EPL>::type xw[kMaxTaps];  // x_{t-3} .. x_t, as loaded
#pragma unroll
      for (int j = 0; j < kMaxTaps; ++j) {
        const int row = te - kMaxTaps + j;
        xw[j] = row >= lo ? ldr<T, EPL>(x + (long)row * CH) : raw_zero<T, EPL>();
      }
      float dsw[kMaxTaps - 1][EPL];  // ds_{t+1}, ds_{t+2}, ds_{t+3}
#pragma unroll
      for (int j = 0; j < kMaxTaps - 1; ++j) zero(dsw[j]);
#pragma unroll 1
      for (int t = te - 1; t >= t0; t -= kBatchBwd) {
        typename Raw<T, EPL>::type graw[kBatchBwd], xnraw[kBatchBwd];
#pragma unroll
        for (int u = 0; u < kBatchBwd; ++u) {
          const int tu = t - u;
          if (tu >= t0) {
            graw[u] = ldr<T, EPL>(dz + (long)tu * CH);
            xnraw[u] = tu - kMaxTaps >= lo ? ldr<T, EPL>(x + (long)(tu - kMaxTaps) * CH) : raw_zero<T, EPL>();
          }
        }
#pragma unroll
        for (int u = 0; u < kBatchBwd; ++u) {
          const int tu = t - u;
          if (tu < t0) break;
          float gr[EPL], xv[kMaxTaps][EPL];
          widen<T, EPL>(graw[u], gr);
#pragma unroll
          for (int j = 0; j < kMaxTaps; ++j) widen<T, EPL>(xw[j], xv[j]);
          float s[EPL], sg[EPL], y[EPL];
          float ss = 0.f, yg = 0.f;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            float v = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxTaps; ++j) v = fmaf(wp[j][e], xv[j][e], v);
            s[e] = v;
            sg[e] = sigmoid(v);
            y[e] = v * sg[e];
            ss = fmaf(y[e], y[e], ss);
            yg = fmaf(y[e], gr[e], yg);
          }
          float ds[EPL];
          if (a.l2norm) {
            const float r = rsqrtf(warp_sum(ss) + a.eps);
            const float c = r * r * warp_sum(yg);
#pragma unroll
            for (int e = 0; e < EPL; ++e) ds[e] = a.scale * r * (gr[e] - y[e] * c);
          } else {
#pragma unroll
            for (int e = 0; e < EPL; ++e) ds[e] = gr[e];
          }
#pragma unroll
          for (int e = 0; e < EPL; ++e) ds[e] *= sg[e] * (1.f + s[e] * (1.f - sg[e]));
          if (tu < t1) {
            float d[EPL];
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
              d[e] = wp[kMaxTaps - 1][e] * ds[e];
#pragma unroll
              for (int j = 0; j < kMaxTaps - 1; ++j) d[e] = fmaf(wp[kMaxTaps - 2 - j][e], dsw[j][e], d[e]);
#pragma unroll
              for (int j = 0; j < kMaxTaps; ++j) dwp[j][e] = fmaf(ds[e], xv[j][e], dwp[j][e]);
            }
            stv<T, EPL>(dx + (long)tu * CH, d);
          }
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            dsw[2][e] = dsw[1][e];
            dsw[1][e] = dsw[0][e];
            dsw[0][e] = ds[e];
          }
          xw[3] = xw[2];
          xw[2] = xw[1];
          xw[1] = xw[0];
          xw[0] = xnraw[u];
        }
      }
      t0 = t1;
    }
  }
  // per-CTA partial dw, unpadded taps: part[blockIdx.x][c][i]
#pragma unroll
  for (int j = 0; j < kMaxTaps; ++j)
#pragma unroll
    for (int e = 0; e < EPL; ++e) red[wi][j][lane * EPL + e] = dwp[j][e];
  __syncthreads();
  float* out = a.part + (long)blockIdx.x * CH * a.W + (long)h * a.D * a.W;
  for (int k = threadIdx.x; k < a.D * a.W; k += blockDim.x) {
    const int c = k / a.W, j = k % a.W + (kMaxTaps - a.W);
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kNbWarps; ++w) v += red[w][j][c];
    out[k] = v;
  }
}

// ---------------------------------------------------------------- partial sums
// out[j] = sum over k of part[k][j] for j < n, k in a fixed order: 32 slices
// of k per column, then the slices in order.
__global__ void __launch_bounds__(1024) sum_partials_kernel(const float* __restrict__ part,
                                                            int nparts, int n,
                                                            float* __restrict__ out) {
  __shared__ float acc[32][33];
  const int j = blockIdx.x * 32 + threadIdx.x;
  float v = 0.f;
  if (j < n)
    for (int k = threadIdx.y; k < nparts; k += 32) v += part[(long)k * n + j];
  acc[threadIdx.y][threadIdx.x] = v;
  __syncthreads();
  if (threadIdx.y == 0 && j < n) {
    float s = 0.f;
    for (int k = 0; k < 32; ++k) s += acc[k][threadIdx.x];
    out[j] = s;
  }
}

// ---------------------------------------------------------------- gated RMS norm
struct NormArgs {
  const void* o;
  const void* gate;
  const float* weight;
  void* out;
  const void* dout;
  void* dO;
  void* dgate;
  float* part;  // backward: [gridDim.x][D] partial dweight
  long rows;
  int D;
  float eps;
};

template <typename T, int EPL>
__global__ void __launch_bounds__(32 * kNbWarps, 2) gated_rmsnorm_fwd_kernel(NormArgs a) {
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int c0 = lane * EPL;
  float wt[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) wt[e] = a.weight[c0 + e];
  const float invD = 1.f / (float)a.D;
  const T* __restrict__ o = static_cast<const T*>(a.o) + c0;
  const T* __restrict__ gate = static_cast<const T*>(a.gate) + c0;
  T* __restrict__ out = static_cast<T*>(a.out) + c0;
  const long step = (long)gridDim.x * kNbWarps * kNormRows;
#pragma unroll 1
  for (long r0 = ((long)blockIdx.x * kNbWarps + wi) * kNormRows; r0 < a.rows; r0 += step) {
    typename Raw<T, EPL>::type oraw[kNormRows], graw[kNormRows];
#pragma unroll
    for (int u = 0; u < kNormRows; ++u)
      if (r0 + u < a.rows) {
        oraw[u] = ldr<T, EPL>(o + r0 * a.D + u * a.D);
        graw[u] = ldr<T, EPL>(gate + r0 * a.D + u * a.D);
      }
#pragma unroll
    for (int u = 0; u < kNormRows; ++u) {
      if (r0 + u >= a.rows) break;
      float ov[EPL], gv[EPL];
      widen<T, EPL>(oraw[u], ov);
      widen<T, EPL>(graw[u], gv);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) ss = fmaf(ov[e], ov[e], ss);
      const float r = rsqrtf(warp_sum(ss) * invD + a.eps);
      float y[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) y[e] = ov[e] * r * wt[e] * (gv[e] * sigmoid(gv[e]));
      stv<T, EPL>(out + r0 * a.D + u * a.D, y);
    }
  }
}

template <typename T, int EPL>
__global__ void __launch_bounds__(32 * kNbWarps, 2) gated_rmsnorm_bwd_kernel(NormArgs a) {
  __shared__ float red[kNbWarps][128];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
  const int c0 = lane * EPL;
  float wt[EPL], dwt[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    wt[e] = a.weight[c0 + e];
    dwt[e] = 0.f;
  }
  const float invD = 1.f / (float)a.D;
  const T* __restrict__ o = static_cast<const T*>(a.o) + c0;
  const T* __restrict__ gate = static_cast<const T*>(a.gate) + c0;
  const T* __restrict__ dout = static_cast<const T*>(a.dout) + c0;
  T* __restrict__ dO = static_cast<T*>(a.dO) + c0;
  T* __restrict__ dgate = static_cast<T*>(a.dgate) + c0;
  const long step = (long)gridDim.x * kNbWarps * kNormRowsBwd;
#pragma unroll 1
  for (long r0 = ((long)blockIdx.x * kNbWarps + wi) * kNormRowsBwd; r0 < a.rows; r0 += step) {
    typename Raw<T, EPL>::type oraw[kNormRowsBwd], graw[kNormRowsBwd], draw[kNormRowsBwd];
#pragma unroll
    for (int u = 0; u < kNormRowsBwd; ++u)
      if (r0 + u < a.rows) {
        const long off = r0 * a.D + u * a.D;
        oraw[u] = ldr<T, EPL>(o + off);
        graw[u] = ldr<T, EPL>(gate + off);
        draw[u] = ldr<T, EPL>(dout + off);
      }
#pragma unroll
    for (int u = 0; u < kNormRowsBwd; ++u) {
      if (r0 + u >= a.rows) break;
      float ov[EPL], gv[EPL], dv[EPL];
      widen<T, EPL>(oraw[u], ov);
      widen<T, EPL>(graw[u], gv);
      widen<T, EPL>(draw[u], dv);
      float ss = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) ss = fmaf(ov[e], ov[e], ss);
      const float r = rsqrtf(warp_sum(ss) * invD + a.eps);
      float n[EPL], sg[EPL], dn[EPL];
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        n[e] = ov[e] * r;
        sg[e] = sigmoid(gv[e]);
        const float act = gv[e] * sg[e];
        dn[e] = dv[e] * wt[e] * act;
        dot = fmaf(dn[e], n[e], dot);
        dwt[e] = fmaf(dv[e] * n[e], act, dwt[e]);
      }
      const float c = warp_sum(dot) * invD;
      float d_o[EPL], d_g[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        d_o[e] = r * (dn[e] - n[e] * c);
        d_g[e] = dv[e] * n[e] * wt[e] * sg[e] * (1.f + gv[e] * (1.f - sg[e]));
      }
      const long off = r0 * a.D + u * a.D;
      stv<T, EPL>(dO + off, d_o);
      stv<T, EPL>(dgate + off, d_g);
    }
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) red[wi][c0 + e] = dwt[e];
  __syncthreads();
  for (int c = threadIdx.x; c < a.D; c += blockDim.x) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kNbWarps; ++w) v += red[w][c];
    a.part[(long)blockIdx.x * a.D + c] = v;
  }
}

// ---------------------------------------------------------------- dispatch
// Grid of the short-conv kernels: x = CTAs per head, y = heads.  The
// backward takes at most about kConvGroupsTarget CTAs in all, each looping
// over an equal share of the run groups (its partial dw is one row of the
// workspace).
int conv_groups(const ConvProblem& p) {
  const long ttot = (long)p.B * p.T;  // at most 2^30 (checked by the caller)
  return (int)((ttot + (long)kRun * kNbWarps - 1) / ((long)kRun * kNbWarps));
}

int conv_bwd_grid_x(const ConvProblem& p) {
  const int groups = conv_groups(p);
  const int cap = std::max(1, kConvGroupsTarget / std::max(1, p.H));
  const int per = (groups + cap - 1) / cap;
  return std::max(1, (groups + per - 1) / per);
}

long norm_row_steps(const NormProblem& p, int rows_per_warp) {
  return (p.rows + (long)kNbWarps * rows_per_warp - 1) / ((long)kNbWarps * rows_per_warp);
}

int norm_bwd_grid_x(const NormProblem& p) {
  const long steps = norm_row_steps(p, kNormRowsBwd);
  const long per = (steps + kNormCtasMax - 1) / kNormCtasMax;
  return (int)std::max(1L, (steps + per - 1) / per);
}

template <typename T, int EPL>
cudaError_t launch_conv(const ConvProblem& p, const ConvArgs& a, bool bwd, cudaStream_t s) {
  const dim3 block(32 * kNbWarps);
  if (!bwd) {
    const dim3 grid(conv_groups(p), p.H);
    prof_before(s);
    if (p.cu_seqlens) short_conv_fwd_kernel<T, EPL, true><<<grid, block, 0, s>>>(a);
    else short_conv_fwd_kernel<T, EPL, false><<<grid, block, 0, s>>>(a);
    prof_after(s, kConvFwd);
    return cudaGetLastError();
  }
  const dim3 grid(conv_bwd_grid_x(p), p.H);
  prof_before(s);
  if (p.cu_seqlens) short_conv_bwd_kernel<T, EPL, true><<<grid, block, 0, s>>>(a);
  else short_conv_bwd_kernel<T, EPL, false><<<grid, block, 0, s>>>(a);
  prof_after(s, kConvBwd);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n = p.H * p.D * p.W;
  prof_before(s);
  sum_partials_kernel<<<(n + 31) / 32, dim3(32, 32), 0, s>>>(a.part, (int)grid.x, n, p.dw);
  prof_after(s, kSumPartials);
  return cudaGetLastError();
}

template <typename T>
cudaError_t conv_dispatch(const ConvProblem& p, const ConvArgs& a, bool bwd, cudaStream_t s) {
  switch (p.D) {
    case 32: return launch_conv<T, 1>(p, a, bwd, s);
    case 64: return launch_conv<T, 2>(p, a, bwd, s);
    default: return launch_conv<T, 4>(p, a, bwd, s);
  }
}

ConvArgs conv_args(const ConvProblem& p) {
  ConvArgs a{};
  a.x = p.x; a.w = p.w; a.z = p.z; a.dz = p.dz; a.dx = p.dx;
  a.part = static_cast<float*>(p.ws);
  a.cu = p.cu_seqlens;
  a.nseq = p.nseq;
  a.T = p.T;
  a.Ttot = p.B * p.T;
  a.H = p.H; a.D = p.D; a.W = p.W;
  a.scale = p.scale; a.eps = p.eps;
  a.l2norm = p.l2norm ? 1 : 0;
  return a;
}

template <typename T, int EPL>
cudaError_t launch_norm(const NormProblem& p, const NormArgs& a, bool bwd, cudaStream_t s) {
  const dim3 block(32 * kNbWarps);
  if (!bwd) {
    const long steps = norm_row_steps(p, kNormRows);
    const int grid = (int)std::min(steps, 65535L * 32);
    prof_before(s);
    gated_rmsnorm_fwd_kernel<T, EPL><<<grid, block, 0, s>>>(a);
    prof_after(s, kNormFwd);
    return cudaGetLastError();
  }
  const int grid = norm_bwd_grid_x(p);
  prof_before(s);
  gated_rmsnorm_bwd_kernel<T, EPL><<<grid, block, 0, s>>>(a);
  prof_after(s, kNormBwd);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  prof_before(s);
  sum_partials_kernel<<<(p.D + 31) / 32, dim3(32, 32), 0, s>>>(a.part, grid, p.D, p.dweight);
  prof_after(s, kSumPartials);
  return cudaGetLastError();
}

template <typename T>
cudaError_t norm_dispatch(const NormProblem& p, const NormArgs& a, bool bwd, cudaStream_t s) {
  switch (p.D) {
    case 32: return launch_norm<T, 1>(p, a, bwd, s);
    case 64: return launch_norm<T, 2>(p, a, bwd, s);
    default: return launch_norm<T, 4>(p, a, bwd, s);
  }
}

NormArgs norm_args(const NormProblem& p) {
  NormArgs a{};
  a.o = p.o; a.gate = p.gate; a.weight = p.weight; a.out = p.out;
  a.dout = p.dout; a.dO = p.dO; a.dgate = p.dgate;
  a.part = static_cast<float*>(p.ws);
  a.rows = p.rows;
  a.D = p.D;
  a.eps = p.eps;
  return a;
}

}  // namespace

size_t short_conv_bwd_workspace(const ConvProblem& p) {
  if ((long)p.B * p.T == 0 || p.H == 0) return 0;
  return align_up((size_t)conv_bwd_grid_x(p) * p.H * p.D * p.W * sizeof(float), 256);
}

cudaError_t short_conv_fwd(const ConvProblem& p, cudaStream_t s) {
  const ConvArgs a = conv_args(p);
  return p.bf16 ? conv_dispatch<__nv_bfloat16>(p, a, false, s) : conv_dispatch<float>(p, a, false, s);
}

cudaError_t short_conv_bwd(const ConvProblem& p, cudaStream_t s) {
  const ConvArgs a = conv_args(p);
  return p.bf16 ? conv_dispatch<__nv_bfloat16>(p, a, true, s) : conv_dispatch<float>(p, a, true, s);
}

size_t gated_rmsnorm_bwd_workspace(const NormProblem& p) {
  if (p.rows == 0) return 0;
  return align_up((size_t)norm_bwd_grid_x(p) * p.D * sizeof(float), 256);
}

cudaError_t gated_rmsnorm_fwd(const NormProblem& p, cudaStream_t s) {
  const NormArgs a = norm_args(p);
  return p.bf16 ? norm_dispatch<__nv_bfloat16>(p, a, false, s) : norm_dispatch<float>(p, a, false, s);
}

cudaError_t gated_rmsnorm_bwd(const NormProblem& p, cudaStream_t s) {
  const NormArgs a = norm_args(p);
  return p.bf16 ? norm_dispatch<__nv_bfloat16>(p, a, true, s) : norm_dispatch<float>(p, a, true, s);
}

cudaError_t nb_read_and_clear_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_nb_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero_word = 0;
  e = cudaMemcpyToSymbol(g_nb_status, &zero_word, sizeof(int));
  if (e != cudaSuccess) return e;
  *status = v;
  return cudaSuccess;
}

}  // namespace gdn
