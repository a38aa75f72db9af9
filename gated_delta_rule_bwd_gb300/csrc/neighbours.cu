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
// Data movement: every warp streams its work through a private ring of
// shared-memory stages filled by TMA copies that complete on one mbarrier per
// stage (a 2-D tensor copy of a chunk's rows of one head for the short conv, a
// 1-D bulk copy of a block of rows for the norm); the warp issues the copies of the
// stage after next before it computes on the current one, so each SM keeps
// 100-200 KB of loads in flight with no register cost and no block-wide
// barrier.  Work items are numbered head-fastest, so the warps running at
// any moment read whole token rows (every head of neighbouring tokens).
//
// Short conv: a warp's item is one head over a run of tokens, cut into
// chunks of TC tokens; a chunk's stage holds its x rows and the three rows
// before them, so every token reads x_{t-3..t} from shared memory (rows
// before the token's sequence start count as zero).  The backward walks its
// item downwards, recomputing s from x (no saved activations), with ds of
// the next three tokens in registers: dx_t = sum_i w_i ds_{t+W-1-i}; an item
// also computes ds for the three tokens after it (a halo that it does not
// store).  dw is summed per warp in registers over its items (all of one
// head), per CTA in shared memory, and over CTAs by a second kernel in a
// fixed order, so the result is bit-for-bit reproducible.
//
// Gated norm: a warp's item is a block of consecutive rows (one bulk copy per
// tensor); dweight is reduced like dw.

#include <algorithm>
#include <map>
#include <mutex>
#include <type_traits>

#include "gdn.h"
#include "gdn_internal.cuh"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace {

__device__ int g_nb_status = 0;

constexpr int kMaxWarps = 16;       // warps per CTA (one CTA per SM)
constexpr int kMaxTaps = 4;         // widest convolution
constexpr int kRingBytes = 200 * 1024;  // shared memory of the staging rings per CTA
constexpr int kStageTarget = 2048;  // bytes of one tensor's rows per stage (about)
constexpr uint32_t kWaitTries = 100000;  // bounded mbarrier waits (about 2 s)

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

// ---------------------------------------------------------------- lane arithmetic
// The kernels are instruction-bound, so element-wise arithmetic on a lane's
// EPL values runs on packed fp32 pairs (FFMA2 / FMUL2 / FADD2: two results
// per instruction, each rounded as the scalar operation would be), and the
// sigmoid uses the hardware 2^x and reciprocal approximations directly:
// sigmoid(x) = 1 / (1 + 2^(-x log2 e)), relative error a few 1e-7, with
// 2^(...) = inf giving 0 and 0 giving 1 at the ends of the range.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float rsqrt_approx(float x) {
  float y;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr float kLog2e = 1.4426950408889634f;

template <int N>
__device__ __forceinline__ void vmul(float (&d)[N], const float (&a)[N], const float (&b)[N]) {
  if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 r = __fmul2_rn(make_float2(a[i], a[i + 1]), make_float2(b[i], b[i + 1]));
      d[i] = r.x;
      d[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = a[i] * b[i];
  }
}

template <int N>
__device__ __forceinline__ void vscale(float (&d)[N], const float (&a)[N], float s) {
  if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 r = __fmul2_rn(make_float2(a[i], a[i + 1]), make_float2(s, s));
      d[i] = r.x;
      d[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = a[i] * s;
  }
}

template <int N>
__device__ __forceinline__ void vfma(float (&d)[N], const float (&a)[N], const float (&b)[N],
                                     const float (&c)[N]) {
  if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 r = __ffma2_rn(make_float2(a[i], a[i + 1]), make_float2(b[i], b[i + 1]),
                                  make_float2(c[i], c[i + 1]));
      d[i] = r.x;
      d[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = fmaf(a[i], b[i], c[i]);
  }
}

// d = a s + c (s broadcast)
template <int N>
__device__ __forceinline__ void vfma_s(float (&d)[N], const float (&a)[N], float s,
                                       const float (&c)[N]) {
  if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 r = __ffma2_rn(make_float2(a[i], a[i + 1]), make_float2(s, s),
                                  make_float2(c[i], c[i + 1]));
      d[i] = r.x;
      d[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = fmaf(a[i], s, c[i]);
  }
}

template <int N>
__device__ __forceinline__ void vadd(float (&d)[N], const float (&a)[N], const float (&b)[N]) {
  if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 r = __fadd2_rn(make_float2(a[i], a[i + 1]), make_float2(b[i], b[i + 1]));
      d[i] = r.x;
      d[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = a[i] + b[i];
  }
}

template <int N>
__device__ __forceinline__ void vadd_s(float (&d)[N], const float (&a)[N], float s) {
  if constexpr (N % 2 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 2) {
      const float2 r = __fadd2_rn(make_float2(a[i], a[i + 1]), make_float2(s, s));
      d[i] = r.x;
      d[i + 1] = r.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < N; ++i) d[i] = a[i] + s;
  }
}

// sum_i a_i b_i over the lane's values
template <int N>
__device__ __forceinline__ float vdot(const float (&a)[N], const float (&b)[N]) {
  if constexpr (N % 2 == 0) {
    float2 acc = __fmul2_rn(make_float2(a[0], a[1]), make_float2(b[0], b[1]));
#pragma unroll
    for (int i = 2; i < N; i += 2)
      acc = __ffma2_rn(make_float2(a[i], a[i + 1]), make_float2(b[i], b[i + 1]), acc);
    return acc.x + acc.y;
  } else {
    float acc = a[0] * b[0];
#pragma unroll
    for (int i = 1; i < N; ++i) acc = fmaf(a[i], b[i], acc);
    return acc;
  }
}

template <int N>
__device__ __forceinline__ void vsigmoid(float (&sg)[N], const float (&x)[N]) {
  float t[N];
  vscale(t, x, -kLog2e);
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = ex2_approx(t[i]);
  vadd_s(t, t, 1.f);
#pragma unroll
  for (int i = 0; i < N; ++i) sg[i] = rcp_approx(t[i]);
}

// ---------------------------------------------------------------- staging
using tc::fence_async_shared;
using tc::fence_barrier_init;
using tc::mbar_arrive_expect_tx;
using tc::mbar_init;
using tc::mbar_wait;
using tc::smem_u32;

// 1-D bulk copy global -> shared completing on `bar` (16-byte aligned
// addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2-D tensor copy of the box at (c0 = channel, c1 = row) into shared memory
// (128-byte aligned), completing on `bar`; rows outside the tensor read as zero.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* tmap, uint64_t* bar, int c0,
                                            int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void report_timeout() { atomicExch(&g_nb_status, GDN_ERR_DEVICE_TIMEOUT); }

// One warp's ring: nstg stages of `bytes` each and one mbarrier per stage.
struct Ring {
  unsigned char* buf;
  uint64_t* full;
  int bytes, nstg;
  __device__ unsigned char* stage(int s) const { return buf + (size_t)s * bytes; }
};

// Carves warp wi's ring out of the dynamic shared memory and initialises its
// barriers (lane 0); the warp syncs before use.
__device__ __forceinline__ Ring make_ring(unsigned char* smem, int nw, int wi, int stage_bytes,
                                          int nstg) {
  Ring r;
  smem += (128 - (smem_u32(smem) & 127)) & 127;  // TMA destinations: 128-byte aligned
  r.buf = smem + (size_t)wi * nstg * stage_bytes;
  r.full = reinterpret_cast<uint64_t*>(smem + (size_t)nw * nstg * stage_bytes) + wi * nstg;
  r.bytes = stage_bytes;
  r.nstg = nstg;
  if ((threadIdx.x & 31) == 0) {
    for (int s = 0; s < nstg; ++s) mbar_init(&r.full[s], 1);
    fence_barrier_init();
  }
  __syncwarp();
  return r;
}

// After a timed-out wait: wait (bounded) for the copies still in flight into
// stages [k, k + inflight) so that none lands after the CTA has exited.
__device__ __forceinline__ void drain(const Ring& r, int k, int inflight) {
  for (int j = 0; j < inflight; ++j) {
    const int kk = k + j;
    mbar_wait(&r.full[kk % r.nstg], (kk / r.nstg) & 1, kWaitTries);
  }
}

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
  float* part;  // backward: partial dw (see conv_partials)
  const int* cu;
  int nseq;
  int T;        // tokens per row (fixed length)
  int Ttot;     // all tokens (at most 2^30)
  int H, D, W;
  float scale, eps;
  int l2norm;
  // work split (host): items are (head, part) pairs numbered head-fastest,
  // part p covering tokens [p L, (p + 1) L); warp gw takes items gw, gw + Wt, ...
  int L, nitems, Wt;
  int TC;       // tokens per chunk
  int nstg, stage_bytes;
  int dz_off;   // backward: stage offset of the dz box (128-byte aligned)
  int cta_heads;  // backward: heads per CTA row of the partials (H when H | warps per CTA)
};

// Items of one warp, cut into chunks of at most TC tokens.  Forward: chunks
// in rising order over [t0, t1).  Backward: chunks in falling order over
// [t0, te), te = min(t1 + 3, Ttot) (the own tokens and the ds halo).
template <bool Bwd>
struct ChunkIter {
  int item, h, t0, t1, te, a, b;  // current chunk [a, b)
  bool valid;
  __device__ void setup(const ConvArgs& p) {
    valid = false;
    for (; item < p.nitems; item += p.Wt) {
      h = item % p.H;
      t0 = (item / p.H) * p.L;
      t1 = min(t0 + p.L, p.Ttot);
      if (t0 >= t1) continue;
      te = min(t1 + kMaxTaps - 1, p.Ttot);
      if (Bwd) {
        b = te;
        a = max(b - p.TC, t0);
      } else {
        a = t0;
        b = min(a + p.TC, t1);
      }
      valid = true;
      return;
    }
  }
  __device__ void init(const ConvArgs& p, int gw) {
    item = gw;
    setup(p);
  }
  __device__ void next(const ConvArgs& p) {
    if (Bwd) {
      if (a > t0) {
        b = a;
        a = max(b - p.TC, t0);
        return;
      }
    } else if (b < t1) {
      a = b;
      b = min(a + p.TC, t1);
      return;
    }
    item += p.Wt;
    setup(p);
  }
};

// Issues one chunk's copies into stage s: the x box of rows [a - 3, a + TC)
// (rows outside the tensor read as zero and are never used) and, backward,
// the dz box of rows [a, a + TC) at dz_off.  Stage row r is global row
// a - 3 + r; only rows below b are used.
template <bool Bwd>
__device__ __forceinline__ void issue_chunk(const ConvArgs& p, const Ring& ring, int s,
                                            const ChunkIter<Bwd>& c, const CUtensorMap* tmx,
                                            const CUtensorMap* tmdz, int rowb) {
  if ((threadIdx.x & 31) == 0) {
    const uint32_t bytes = (p.TC + kMaxTaps - 1 + (Bwd ? p.TC : 0)) * rowb;
    mbar_arrive_expect_tx(&ring.full[s], bytes);
    tma_load_2d(ring.stage(s), tmx, &ring.full[s], c.h * p.D, c.a - (kMaxTaps - 1));
    if (Bwd) tma_load_2d(ring.stage(s) + p.dz_off, tmdz, &ring.full[s], c.h * p.D, c.a);
  }
  __syncwarp();
}

// ---------------------------------------------------------------- short conv forward
// x_{t-3..t} of the lane's channels from the chunk's stage (rows below lo,
// the token's sequence start, read as zero unless Fast says none is).
template <typename T, int EPL, bool Fast>
__device__ __forceinline__ void load_window(const unsigned char* xs, int xb, int rowb, int t, int lo,
                                            float (&xv)[kMaxTaps][EPL]) {
#pragma unroll
  for (int j = 0; j < kMaxTaps; ++j) {
    const int row = t - (kMaxTaps - 1) + j;
    if (Fast || row >= lo)
      widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(xs + (row - xb) * rowb),
                    xv[j]);
    else
      zero(xv[j]);
  }
}

// One token of the forward from its window x_{t-3..t}: z = SiLU(sum_j wp_j
// x_{t-3+j}), L2-normalised per head and scaled.
template <typename T, int EPL, bool Norm>
__device__ __forceinline__ void conv_fwd_from(const float (&x0)[EPL], const float (&x1)[EPL],
                                              const float (&x2)[EPL], const float (&x3)[EPL],
                                              const float (&wp)[kMaxTaps][EPL], float scale,
                                              float eps, T* __restrict__ zrow) {
  float sv[EPL], sg[EPL], y[EPL];
  vmul(sv, wp[3], x3);
  vfma(sv, wp[2], x2, sv);
  vfma(sv, wp[1], x1, sv);
  vfma(sv, wp[0], x0, sv);
  vsigmoid(sg, sv);
  vmul(y, sv, sg);
  if (Norm) vscale(y, y, scale * rsqrt_approx(warp_sum(vdot(y, y)) + eps));
  stv<T, EPL>(zrow, y);
}

template <typename T, int EPL>
__device__ __forceinline__ void smem_row(const unsigned char* xs, int rowb, int r, float (&v)[EPL]) {
  widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(xs + r * rowb), v);
}

// One token with sequence checks: rows before lo read as zero.
template <typename T, int EPL, bool Norm>
__device__ __forceinline__ void conv_fwd_token(const unsigned char* xs, int xb, int rowb, int t,
                                               int lo, const float (&wp)[kMaxTaps][EPL],
                                               float scale, float eps, T* __restrict__ zrow) {
  float xv[kMaxTaps][EPL];
  load_window<T, EPL, false>(xs, xb, rowb, t, lo, xv);
  conv_fwd_from<T, EPL, Norm>(xv[0], xv[1], xv[2], xv[3], wp, scale, eps, zrow);
}

// Four tokens t..t+3 of one sequence: their seven rows x_{t-3..t+3} are read once.
template <typename T, int EPL, bool Norm>
__device__ __forceinline__ void conv_fwd_group(const unsigned char* xs, int xb, int rowb, int t,
                                               const float (&wp)[kMaxTaps][EPL], float scale,
                                               float eps, T* __restrict__ z, long CH) {
  float xr[7][EPL];
#pragma unroll
  for (int r = 0; r < 7; ++r) smem_row<T, EPL>(xs, rowb, t - (kMaxTaps - 1) + r - xb, xr[r]);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    conv_fwd_from<T, EPL, Norm>(xr[q], xr[q + 1], xr[q + 2], xr[q + 3], wp, scale, eps,
                                z + (long)(t + q) * CH);
}

template <typename T, int EPL, bool Packed, bool Norm>
__global__ void __launch_bounds__(32 * kMaxWarps, 1)
short_conv_fwd_kernel(const __grid_constant__ CUtensorMap tmx, ConvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (Packed && blockIdx.x == 0) check_offsets(a.cu, a.nseq, a.Ttot);
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const Ring ring = make_ring(smem, nw, wi, a.stage_bytes, a.nstg);
  const int gw = blockIdx.x * nw + wi;
  const int rowb = a.D * (int)sizeof(T);
  const long CH = (long)a.H * a.D;
  ChunkIter<false> pc, cc;
  pc.init(a, gw);
  cc = pc;
  int issued = 0;
  for (; issued < a.nstg && pc.valid; ++issued, pc.next(a))
    issue_chunk<false>(a, ring, issued, pc, &tmx, &tmx, rowb);
  int h = -1;
  float wp[kMaxTaps][EPL];
  for (int k = 0; cc.valid; ++k, cc.next(a)) {
    const int s = k % a.nstg;
    if (!mbar_wait(&ring.full[s], (k / a.nstg) & 1, kWaitTries)) {
      if (lane == 0) report_timeout();
      drain(ring, k + 1, issued - k - 1);
      return;
    }
    if (cc.h != h) {
      h = cc.h;
      load_taps<EPL>(a.w, a.W, h * a.D + lane * EPL, wp);
    }
    const unsigned char* xs = ring.stage(s) + lane * EPL * (int)sizeof(T);
    const int xb = cc.a - (kMaxTaps - 1);  // global row of stage row 0
    T* __restrict__ z = static_cast<T*>(a.z) + h * a.D + lane * EPL;
    int lo, hi;
    seq_bounds<Packed>(cc.a, a.T, a.Ttot, a.cu, a.nseq, lo, hi);
    int t = cc.a;
    if (lo <= xb && hi >= cc.b) {
      // no sequence start among the chunk's rows: four independent tokens at a time
      for (; t + 4 <= cc.b; t += 4) conv_fwd_group<T, EPL, Norm>(xs, xb, rowb, t, wp, a.scale, a.eps, z, CH);
      for (; t < cc.b; ++t)
        conv_fwd_token<T, EPL, Norm>(xs, xb, rowb, t, lo, wp, a.scale, a.eps, z + (long)t * CH);
    } else {
      for (; t < cc.b; ++t) {
        if (t >= hi) seq_bounds<Packed>(t, a.T, a.Ttot, a.cu, a.nseq, lo, hi);
        conv_fwd_token<T, EPL, Norm>(xs, xb, rowb, t, lo, wp, a.scale, a.eps, z + (long)t * CH);
      }
    }
    __syncwarp();
    fence_async_shared();
    if (pc.valid) {
      issue_chunk<false>(a, ring, s, pc, &tmx, &tmx, rowb);
      pc.next(a);
      ++issued;
    }
  }
}

// ---------------------------------------------------------------- short conv backward
// ds_t of one token from its window x_{t-3..t} and dz_t: the gradient at the
// pre-activation s_t (through the L2 norm and SiLU); own tokens add
// ds_t x_{t-3+j} to dw.
template <typename T, int EPL, bool Norm>
__device__ __forceinline__ void conv_bwd_from(const float (&x0)[EPL], const float (&x1)[EPL],
                                              const float (&x2)[EPL], const float (&x3)[EPL],
                                              const float (&gr)[EPL], bool own,
                                              const float (&wp)[kMaxTaps][EPL], float scale,
                                              float eps, float (&ds)[EPL],
                                              float (&dwp)[kMaxTaps][EPL]) {
  float sv[EPL], sg[EPL], y[EPL], dy[EPL];
  vmul(sv, wp[3], x3);
  vfma(sv, wp[2], x2, sv);
  vfma(sv, wp[1], x1, sv);
  vfma(sv, wp[0], x0, sv);
  vsigmoid(sg, sv);
  vmul(y, sv, sg);
  if (Norm) {
    const float r = rsqrt_approx(warp_sum(vdot(y, y)) + eps);
    const float c = r * r * warp_sum(vdot(y, gr));
    vfma_s(dy, y, -c, gr);     // g - c y
    vscale(dy, dy, scale * r);
  } else {
#pragma unroll
    for (int e = 0; e < EPL; ++e) dy[e] = gr[e];
  }
  // SiLU'(s) = sg (1 + s (1 - sg)) = (y + sg) - y sg
  float ysg[EPL], d1[EPL];
  vmul(ysg, y, sg);
  vadd(d1, y, sg);
  vfma_s(d1, ysg, -1.f, d1);
  vmul(ds, dy, d1);
  if (own) {
    vfma(dwp[0], ds, x0, dwp[0]);
    vfma(dwp[1], ds, x1, dwp[1]);
    vfma(dwp[2], ds, x2, dwp[2]);
    vfma(dwp[3], ds, x3, dwp[3]);
  }
}

template <typename T, int EPL, bool Norm>
__device__ __forceinline__ void conv_bwd_ds(const unsigned char* xs, const unsigned char* dzs,
                                            int xb, int a0, int rowb, int t, int lo, bool own,
                                            const float (&wp)[kMaxTaps][EPL], float scale,
                                            float eps, float (&ds)[EPL],
                                            float (&dwp)[kMaxTaps][EPL]) {
  float gr[EPL], xv[kMaxTaps][EPL];
  load_window<T, EPL, false>(xs, xb, rowb, t, lo, xv);
  smem_row<T, EPL>(dzs, rowb, t - a0, gr);
  conv_bwd_from<T, EPL, Norm>(xv[0], xv[1], xv[2], xv[3], gr, own, wp, scale, eps, ds, dwp);
}

// dx_t = sum_j wp_j ds_{t+3-j} from ds_t and the window of later ds (own
// tokens only); then the window moves down one token.
template <typename T, int EPL>
__device__ __forceinline__ void conv_bwd_finish(bool own, const float (&wp)[kMaxTaps][EPL],
                                                const float (&ds)[EPL],
                                                float (&dsw)[kMaxTaps - 1][EPL],
                                                T* __restrict__ dxrow) {
  if (own) {
    float d[EPL];
    vmul(d, wp[3], ds);
    vfma(d, wp[2], dsw[0], d);
    vfma(d, wp[1], dsw[1], d);
    vfma(d, wp[0], dsw[2], d);
    stv<T, EPL>(dxrow, d);
  }
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    dsw[2][e] = dsw[1][e];
    dsw[1][e] = dsw[0][e];
    dsw[0][e] = ds[e];
  }
}

template <typename T, int EPL, bool Packed, bool Norm>
__global__ void __launch_bounds__(32 * kMaxWarps, 1)
short_conv_bwd_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmdz,
                      ConvArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  if (Packed && blockIdx.x == 0) check_offsets(a.cu, a.nseq, a.Ttot);
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const Ring ring = make_ring(smem, nw, wi, a.stage_bytes, a.nstg);
  const int gw = blockIdx.x * nw + wi;
  const int rowb = a.D * (int)sizeof(T);
  const long CH = (long)a.H * a.D;
  ChunkIter<true> pc, cc;
  pc.init(a, gw);
  cc = pc;
  const int h = cc.valid ? cc.h : -1;  // every item of a warp has the same head (Wt % H == 0)
  float wp[kMaxTaps][EPL], dwp[kMaxTaps][EPL];
  if (h >= 0) load_taps<EPL>(a.w, a.W, h * a.D + lane * EPL, wp);
#pragma unroll
  for (int j = 0; j < kMaxTaps; ++j) zero(dwp[j]);
  int issued = 0;
  for (; issued < a.nstg && pc.valid; ++issued, pc.next(a))
    issue_chunk<true>(a, ring, issued, pc, &tmx, &tmdz, rowb);
  int item = -1, lo = 0, hi = 0;
  float dsw[kMaxTaps - 1][EPL];  // ds of the next three tokens (same sequence), else 0
  for (int k = 0; cc.valid; ++k, cc.next(a)) {
    const int s = k % a.nstg;
    if (!mbar_wait(&ring.full[s], (k / a.nstg) & 1, kWaitTries)) {
      if (lane == 0) report_timeout();
      drain(ring, k + 1, issued - k - 1);
      break;
    }
    const unsigned char* xs = ring.stage(s) + lane * EPL * (int)sizeof(T);
    const unsigned char* dzs = xs + a.dz_off;
    const int xb = cc.a - (kMaxTaps - 1);
    T* __restrict__ dx = static_cast<T*>(a.dx) + h * a.D + lane * EPL;
    if (cc.item != item) {  // a new item starts at its top: no later ds
      item = cc.item;
#pragma unroll
      for (int j = 0; j < kMaxTaps - 1; ++j) zero(dsw[j]);
      seq_bounds<Packed>(cc.b - 1, a.T, a.Ttot, a.cu, a.nseq, lo, hi);
    }
    int t = cc.b - 1;
    if (lo <= xb) {
      // the chunk's tokens and rows all lie in one sequence: ds of four
      // tokens at a time, then their dx from the top down
      for (; t - 3 >= cc.a; t -= 4) {
        // tokens t, t-1, t-2, t-3: x rows t-6..t read once
        float ds[4][EPL], xr[7][EPL];
#pragma unroll
        for (int r = 0; r < 7; ++r) smem_row<T, EPL>(xs, rowb, t - 6 + r - xb, xr[r]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float gr[EPL];
          smem_row<T, EPL>(dzs, rowb, t - q - cc.a, gr);
          conv_bwd_from<T, EPL, Norm>(xr[3 - q], xr[4 - q], xr[5 - q], xr[6 - q], gr,
                                      t - q < cc.t1, wp, a.scale, a.eps, ds[q], dwp);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
          conv_bwd_finish<T, EPL>(t - q < cc.t1, wp, ds[q], dsw, dx + (long)(t - q) * CH);
      }
      for (; t >= cc.a; --t) {
        float ds[EPL];
        conv_bwd_ds<T, EPL, Norm>(xs, dzs, xb, cc.a, rowb, t, lo, t < cc.t1, wp, a.scale, a.eps,
                                  ds, dwp);
        conv_bwd_finish<T, EPL>(t < cc.t1, wp, ds, dsw, dx + (long)t * CH);
      }
    } else {
      for (; t >= cc.a; --t) {
        if (t < lo) {  // crossed into the previous sequence
          seq_bounds<Packed>(t, a.T, a.Ttot, a.cu, a.nseq, lo, hi);
#pragma unroll
          for (int j = 0; j < kMaxTaps - 1; ++j) zero(dsw[j]);
        }
        float ds[EPL];
        conv_bwd_ds<T, EPL, Norm>(xs, dzs, xb, cc.a, rowb, t, lo, t < cc.t1, wp, a.scale, a.eps,
                                  ds, dwp);
        conv_bwd_finish<T, EPL>(t < cc.t1, wp, ds, dsw, dx + (long)t * CH);
      }
    }
    __syncwarp();
    fence_async_shared();
    if (pc.valid) {
      issue_chunk<true>(a, ring, s, pc, &tmx, &tmdz, rowb);
      pc.next(a);
      ++issued;
    }
  }
  // partial dw: the CTA's warps sum their registers per head in shared memory
  // (the rings are done), then one row per CTA (cta_heads heads) or per warp
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [nw][D * W]
  const int DW = a.D * a.W;
  if (h >= 0) {
#pragma unroll
    for (int j = 0; j < kMaxTaps; ++j) {
      const int i = j - (kMaxTaps - a.W);
      if (i >= 0)
#pragma unroll
        for (int e = 0; e < EPL; ++e) red[wi * DW + (lane * EPL + e) * a.W + i] = dwp[j][e];
    }
  } else {
    for (int k = lane; k < DW; k += 32) red[wi * DW + k] = 0.f;
  }
  __syncthreads();
  if (a.cta_heads == a.H) {
    // H divides the warps of a CTA: warp w has head w % H; one row per CTA
    float* out = a.part + (long)blockIdx.x * a.H * DW;
    for (int k = threadIdx.x; k < a.H * DW; k += blockDim.x) {
      const int hh = k / DW, c = k % DW;
      float v = 0.f;
      for (int w = hh; w < nw; w += a.H) v += red[w * DW + c];
      out[k] = v;
    }
  } else {
    // one row per warp: warp gw = q H + h writes row q, head h
    for (int k = threadIdx.x; k < nw * DW; k += blockDim.x) {
      const int w = k / DW, c = k % DW;
      const int g = blockIdx.x * nw + w;
      a.part[(long)g * DW + c] = red[w * DW + c];
    }
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
  int RC;       // rows per chunk; warp gw takes chunks gw, gw + Wt, ...
  long nchunks;
  int Wt, nstg, stage_bytes;
};

// Issues chunk ch's rows of `ntens` tensors into stage s (one bulk copy each).
__device__ __forceinline__ void issue_rows(const NormArgs& p, const Ring& ring, int s, long ch,
                                           const void* const* src, int ntens, int rowb) {
  if ((threadIdx.x & 31) != 0) return;
  const long r0 = ch * p.RC;
  const int n = (int)min((long)p.RC, p.rows - r0);
  const uint32_t bytes = (uint32_t)(n * rowb);
  mbar_arrive_expect_tx(&ring.full[s], bytes * ntens);
  for (int i = 0; i < ntens; ++i)
    bulk_copy(ring.stage(s) + i * p.RC * rowb,
              static_cast<const unsigned char*>(src[i]) + r0 * rowb, bytes, &ring.full[s]);
}

// One row of the gated norm: out = o r weight SiLU(gate), r = 1 / sqrt(mean(o^2) + eps).
template <typename T, int EPL>
__device__ __forceinline__ void norm_fwd_row(const unsigned char* os, const unsigned char* gs,
                                             const float (&wt)[EPL], float invD, float eps,
                                             T* __restrict__ out) {
  float ov[EPL], gv[EPL];
  widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(os), ov);
  widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(gs), gv);
  const float r = rsqrt_approx(warp_sum(vdot(ov, ov)) * invD + eps);
  float sg[EPL], act[EPL], wr[EPL], y[EPL];
  vsigmoid(sg, gv);
  vmul(act, gv, sg);  // SiLU(gate)
  vscale(wr, wt, r);
  vmul(y, ov, wr);
  vmul(y, y, act);
  stv<T, EPL>(out, y);
}

// One row of the gated norm's backward: do, dgate, and the row's dweight terms.
template <typename T, int EPL>
__device__ __forceinline__ void norm_bwd_row(const unsigned char* os, const unsigned char* gs,
                                             const unsigned char* ds, const float (&wt)[EPL],
                                             float invD, float eps, float (&dwt)[EPL],
                                             T* __restrict__ dO, T* __restrict__ dgate) {
  float ov[EPL], gv[EPL], dv[EPL];
  widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(os), ov);
  widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(gs), gv);
  widen<T, EPL>(*reinterpret_cast<const typename Raw<T, EPL>::type*>(ds), dv);
  const float r = rsqrt_approx(warp_sum(vdot(ov, ov)) * invD + eps);
  float nrm[EPL], sg[EPL], act[EPL], dn[EPL], dvn[EPL], t[EPL];
  vscale(nrm, ov, r);
  vsigmoid(sg, gv);
  vmul(act, gv, sg);        // SiLU(gate)
  vmul(t, dv, wt);
  vmul(dn, t, act);         // d(out)/d(n) terms: dout weight SiLU(gate)
  vmul(dvn, dv, nrm);
  vfma(dwt, dvn, act, dwt); // dweight += dout n SiLU(gate)
  const float c = warp_sum(vdot(dn, nrm)) * invD;
  float d_o[EPL], d_g[EPL], d1[EPL], as[EPL];
  vfma_s(t, nrm, -c, dn);
  vscale(d_o, t, r);        // do = r (dn - n c)
  // dgate = dout n weight SiLU'(gate), SiLU'(g) = (act + sg) - act sg
  vmul(as, act, sg);
  vadd(d1, act, sg);
  vfma_s(d1, as, -1.f, d1);
  vmul(t, dvn, wt);
  vmul(d_g, t, d1);
  stv<T, EPL>(dO, d_o);
  stv<T, EPL>(dgate, d_g);
}

template <typename T, int EPL>
__global__ void __launch_bounds__(32 * kMaxWarps, 1) gated_rmsnorm_fwd_kernel(NormArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const Ring ring = make_ring(smem, nw, wi, a.stage_bytes, a.nstg);
  const long gw = (long)blockIdx.x * nw + wi;
  const int rowb = a.D * (int)sizeof(T), c0 = lane * EPL;
  const void* src[2] = {a.o, a.gate};
  float wt[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) wt[e] = a.weight[c0 + e];
  const float invD = 1.f / (float)a.D;
  long pch = gw;
  int issued = 0;
  for (; issued < a.nstg && pch < a.nchunks; ++issued, pch += a.Wt)
    issue_rows(a, ring, issued, pch, src, 2, rowb);
  __syncwarp();
  int k = 0;
  for (long ch = gw; ch < a.nchunks; ch += a.Wt, ++k) {
    const int s = k % a.nstg;
    if (!mbar_wait(&ring.full[s], (k / a.nstg) & 1, kWaitTries)) {
      if (lane == 0) report_timeout();
      drain(ring, k + 1, issued - k - 1);
      return;
    }
    const unsigned char* os = ring.stage(s) + c0 * (int)sizeof(T);
    const unsigned char* gs = os + a.RC * rowb;
    const long r0 = ch * a.RC;
    const int n = (int)min((long)a.RC, a.rows - r0);
    T* __restrict__ out = static_cast<T*>(a.out) + r0 * a.D + c0;
    int u = 0;
    for (; u + 4 <= n; u += 4) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        norm_fwd_row<T, EPL>(os + (u + q) * rowb, gs + (u + q) * rowb, wt, invD, a.eps,
                             out + (long)(u + q) * a.D);
    }
    for (; u < n; ++u)
      norm_fwd_row<T, EPL>(os + u * rowb, gs + u * rowb, wt, invD, a.eps, out + (long)u * a.D);
    __syncwarp();
    fence_async_shared();
    if (pch < a.nchunks) {
      issue_rows(a, ring, s, pch, src, 2, rowb);
      __syncwarp();
      pch += a.Wt;
      ++issued;
    }
  }
}

template <typename T, int EPL>
__global__ void __launch_bounds__(32 * kMaxWarps, 1) gated_rmsnorm_bwd_kernel(NormArgs a) {
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const Ring ring = make_ring(smem, nw, wi, a.stage_bytes, a.nstg);
  const long gw = (long)blockIdx.x * nw + wi;
  const int rowb = a.D * (int)sizeof(T), c0 = lane * EPL;
  const void* src[3] = {a.o, a.gate, a.dout};
  float wt[EPL], dwt[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) {
    wt[e] = a.weight[c0 + e];
    dwt[e] = 0.f;
  }
  const float invD = 1.f / (float)a.D;
  long pch = gw;
  int issued = 0;
  for (; issued < a.nstg && pch < a.nchunks; ++issued, pch += a.Wt)
    issue_rows(a, ring, issued, pch, src, 3, rowb);
  __syncwarp();
  int k = 0;
  for (long ch = gw; ch < a.nchunks; ch += a.Wt, ++k) {
    const int s = k % a.nstg;
    if (!mbar_wait(&ring.full[s], (k / a.nstg) & 1, kWaitTries)) {
      if (lane == 0) report_timeout();
      drain(ring, k + 1, issued - k - 1);
      break;
    }
    const unsigned char* os = ring.stage(s) + c0 * (int)sizeof(T);
    const unsigned char* gs = os + a.RC * rowb;
    const unsigned char* dsm = gs + a.RC * rowb;
    const long r0 = ch * a.RC;
    const int n = (int)min((long)a.RC, a.rows - r0);
    T* __restrict__ dO = static_cast<T*>(a.dO) + r0 * a.D + c0;
    T* __restrict__ dgate = static_cast<T*>(a.dgate) + r0 * a.D + c0;
    int u = 0;
    for (; u + 4 <= n; u += 4) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        norm_bwd_row<T, EPL>(os + (u + q) * rowb, gs + (u + q) * rowb, dsm + (u + q) * rowb, wt,
                             invD, a.eps, dwt, dO + (long)(u + q) * a.D, dgate + (long)(u + q) * a.D);
    }
    for (; u < n; ++u)
      norm_bwd_row<T, EPL>(os + u * rowb, gs + u * rowb, dsm + u * rowb, wt, invD, a.eps, dwt,
                           dO + (long)u * a.D, dgate + (long)u * a.D);
    __syncwarp();
    fence_async_shared();
    if (pch < a.nchunks) {
      issue_rows(a, ring, s, pch, src, 3, rowb);
      __syncwarp();
      pch += a.Wt;
      ++issued;
    }
  }
  __syncthreads();
  float* red = reinterpret_cast<float*>(smem);  // [nw][D]
#pragma unroll
  for (int e = 0; e < EPL; ++e) red[wi * a.D + c0 + e] = dwt[e];
  __syncthreads();
  for (int c = threadIdx.x; c < a.D; c += blockDim.x) {
    float v = 0.f;
    for (int w = 0; w < nw; ++w) v += red[w * a.D + c];
    a.part[(long)blockIdx.x * a.D + c] = v;
  }
}

// ---------------------------------------------------------------- launch geometry
int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
      v = 152;
    n = v;
  }
  return n;
}

int gcd(int x, int y) { return y == 0 ? x : gcd(y, x % y); }

// Raises a kernel's dynamic shared-memory limit once per device (the call
// costs host time on every launch otherwise).
cudaError_t set_smem(const void* kf, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = done[{dev, kf}];
  if (have >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kf, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) have = smem;
  return e;
}

// Staging geometry shared by the kernels: warps per CTA, stages, stage bytes.
struct Geometry {
  int nw, nstg, stage_bytes, chunk;  // chunk: tokens (conv) or rows (norm) per stage
  size_t smem() const { return 128 + (size_t)nw * nstg * stage_bytes + (size_t)nw * nstg * 8; }
};

int conv_dz_off(int D, int esize, int chunk) {
  return ((chunk + kMaxTaps - 1) * D * esize + 127) / 128 * 128;
}

// conv: a stage holds chunk + 3 x rows (and, backward, chunk dz rows)
Geometry conv_geometry(int D, int esize, bool bwd) {
  const int rowb = D * esize;
  Geometry g;
  // the forward holds x only: twice the tokens per stage (fewer chunk overheads)
  g.chunk = std::max(bwd ? 8 : 16, (bwd ? kStageTarget : 2 * kStageTarget) / rowb);
  const int bytes = bwd ? conv_dz_off(D, esize, g.chunk) + g.chunk * rowb
                        : (g.chunk + kMaxTaps - 1) * rowb;
  g.stage_bytes = (bytes + 127) / 128 * 128;
  g.nw = kMaxWarps;
  g.nstg = 3;
  while (g.nstg > 2 && g.smem() > (size_t)kRingBytes) --g.nstg;
  while (g.nw > 4 && g.smem() > (size_t)kRingBytes) g.nw /= 2;
  return g;
}

Geometry norm_geometry(int D, int esize, bool bwd) {
  const int rowb = D * esize;
  Geometry g;
  g.chunk = std::max(1, kStageTarget / rowb);
  g.stage_bytes = (bwd ? 3 : 2) * g.chunk * rowb;
  g.nw = kMaxWarps;
  g.nstg = 3;
  while (g.nstg > 2 && g.smem() > (size_t)kRingBytes) --g.nstg;
  while (g.nw > 4 && g.smem() > (size_t)kRingBytes) g.nw /= 2;
  return g;
}

// Conv grid: one CTA per SM; the backward keeps the warp count a multiple of H
// (every warp's items then have one head, so dw stays in its registers).
int conv_grid(const ConvProblem& p, const Geometry& g, bool bwd) {
  int grid = num_sms();
  if (bwd) {
    const int step = p.H / gcd(p.H, g.nw);  // CTAs per multiple of H warps
    grid = std::max(1, grid / step) * step;
  }
  return grid;
}

ConvArgs conv_args(const ConvProblem& p, const Geometry& g, int grid) {
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
  a.Wt = grid * g.nw;
  // about two items per warp: P parts of L tokens per head
  const long P = std::max(1L, ((long)2 * a.Wt + p.H - 1) / p.H);
  a.L = (int)std::max(1L, ((long)a.Ttot + P - 1) / P);
  a.nitems = (int)(((long)a.Ttot + a.L - 1) / a.L) * p.H;
  a.TC = g.chunk;
  a.nstg = g.nstg;
  a.stage_bytes = g.stage_bytes;
  a.dz_off = conv_dz_off(p.D, p.bf16 ? 2 : 4, g.chunk);
  a.cta_heads = (g.nw % p.H == 0) ? p.H : 0;
  return a;
}

// Rows of partial dw: one per CTA (H | warps per CTA) or one per H warps.
int conv_partials(const ConvProblem& p, const Geometry& g, int grid) {
  return (g.nw % p.H == 0) ? grid : grid * g.nw / p.H;
}

// 2-D map over a [Ttot, H*D] token tensor; box = D channels x rows tokens,
// no swizzle; rows outside [0, Ttot) read as zero.
template <typename T>
cudaError_t make_rows_map(CUtensorMap* m, const void* ptr, const ConvProblem& p, int rows) {
  auto enc = tc::get_encoder();
  if (!enc) return cudaErrorNotSupported;
  const CUtensorMapDataType dt =
      std::is_same<T, float>::value ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  cuuint64_t dims[2] = {(cuuint64_t)p.H * p.D, (cuuint64_t)p.B * p.T};
  cuuint64_t strides[1] = {(cuuint64_t)p.H * p.D * sizeof(T)};
  cuuint32_t box[2] = {(cuuint32_t)p.D, (cuuint32_t)rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <typename T, int EPL>
cudaError_t launch_conv(const ConvProblem& p, bool bwd, cudaStream_t s) {
  const Geometry g = conv_geometry(p.D, (int)sizeof(T), bwd);
  const int grid = conv_grid(p, g, bwd);
  const ConvArgs a = conv_args(p, g, grid);
  const size_t smem = std::max(g.smem(), bwd ? (size_t)g.nw * p.D * p.W * 4 : (size_t)0);
  CUtensorMap tmx, tmdz;
  cudaError_t e = make_rows_map<T>(&tmx, p.x, p, g.chunk + kMaxTaps - 1);
  if (e == cudaSuccess && bwd) e = make_rows_map<T>(&tmdz, p.dz, p, g.chunk);
  if (e != cudaSuccess) return e;
  if (bwd) {
    auto kf = p.cu_seqlens ? (p.l2norm ? short_conv_bwd_kernel<T, EPL, true, true>
                                       : short_conv_bwd_kernel<T, EPL, true, false>)
                           : (p.l2norm ? short_conv_bwd_kernel<T, EPL, false, true>
                                       : short_conv_bwd_kernel<T, EPL, false, false>);
    e = set_smem(reinterpret_cast<const void*>(kf), smem);
    if (e != cudaSuccess) return e;
    prof_before(s);
    kf<<<grid, 32 * g.nw, smem, s>>>(tmx, tmdz, a);
    prof_after(s, kConvBwd);
  } else {
    auto kf = p.cu_seqlens ? (p.l2norm ? short_conv_fwd_kernel<T, EPL, true, true>
                                       : short_conv_fwd_kernel<T, EPL, true, false>)
                           : (p.l2norm ? short_conv_fwd_kernel<T, EPL, false, true>
                                       : short_conv_fwd_kernel<T, EPL, false, false>);
    e = set_smem(reinterpret_cast<const void*>(kf), smem);
    if (e != cudaSuccess) return e;
    prof_before(s);
    kf<<<grid, 32 * g.nw, smem, s>>>(tmx, a);
    prof_after(s, kConvFwd);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess || !bwd) return e;
  const int n = p.H * p.D * p.W;
  prof_before(s);
  sum_partials_kernel<<<(n + 31) / 32, dim3(32, 32), 0, s>>>(a.part, conv_partials(p, g, grid), n,
                                                             p.dw);
  prof_after(s, kSumPartials);
  return cudaGetLastError();
}

template <typename T>
cudaError_t conv_dispatch(const ConvProblem& p, bool bwd, cudaStream_t s) {
  switch (p.D) {
    case 32: return launch_conv<T, 1>(p, bwd, s);
    case 64: return launch_conv<T, 2>(p, bwd, s);
    default: return launch_conv<T, 4>(p, bwd, s);
  }
}

int norm_grid(const NormProblem& p, const Geometry& g) {
  const long chunks = (p.rows + g.chunk - 1) / g.chunk;
  const long ctas = (chunks + g.nw - 1) / g.nw;
  return (int)std::max(1L, std::min((long)num_sms(), ctas));
}

template <typename T, int EPL>
cudaError_t launch_norm(const NormProblem& p, bool bwd, cudaStream_t s) {
  const Geometry g = norm_geometry(p.D, (int)sizeof(T), bwd);
  const int grid = norm_grid(p, g);
  NormArgs a{};
  a.o = p.o; a.gate = p.gate; a.weight = p.weight; a.out = p.out;
  a.dout = p.dout; a.dO = p.dO; a.dgate = p.dgate;
  a.part = static_cast<float*>(p.ws);
  a.rows = p.rows;
  a.D = p.D;
  a.eps = p.eps;
  a.RC = g.chunk;
  a.nchunks = (p.rows + g.chunk - 1) / g.chunk;
  a.Wt = grid * g.nw;
  a.nstg = g.nstg;
  a.stage_bytes = g.stage_bytes;
  const size_t smem = std::max(g.smem(), bwd ? (size_t)g.nw * p.D * 4 : (size_t)0);
  auto kf = bwd ? gated_rmsnorm_bwd_kernel<T, EPL> : gated_rmsnorm_fwd_kernel<T, EPL>;
  cudaError_t e = set_smem(reinterpret_cast<const void*>(kf), smem);
  if (e != cudaSuccess) return e;
  prof_before(s);
  kf<<<grid, 32 * g.nw, smem, s>>>(a);
  prof_after(s, bwd ? kNormBwd : kNormFwd);
  e = cudaGetLastError();
  if (e != cudaSuccess || !bwd) return e;
  prof_before(s);
  sum_partials_kernel<<<(p.D + 31) / 32, dim3(32, 32), 0, s>>>(a.part, grid, p.D, p.dweight);
  prof_after(s, kSumPartials);
  return cudaGetLastError();
}

template <typename T>
cudaError_t norm_dispatch(const NormProblem& p, bool bwd, cudaStream_t s) {
  switch (p.D) {
    case 32: return launch_norm<T, 1>(p, bwd, s);
    case 64: return launch_norm<T, 2>(p, bwd, s);
    default: return launch_norm<T, 4>(p, bwd, s);
  }
}

}  // namespace

size_t short_conv_bwd_workspace(const ConvProblem& p) {
  if ((long)p.B * p.T == 0 || p.H == 0) return 0;
  const Geometry g = conv_geometry(p.D, p.bf16 ? 2 : 4, true);
  const int grid = conv_grid(p, g, true);
  return align_up((size_t)conv_partials(p, g, grid) * p.H * p.D * p.W * sizeof(float), 256);
}

cudaError_t short_conv_fwd(const ConvProblem& p, cudaStream_t s) {
  return p.bf16 ? conv_dispatch<__nv_bfloat16>(p, false, s) : conv_dispatch<float>(p, false, s);
}

cudaError_t short_conv_bwd(const ConvProblem& p, cudaStream_t s) {
  return p.bf16 ? conv_dispatch<__nv_bfloat16>(p, true, s) : conv_dispatch<float>(p, true, s);
}

size_t gated_rmsnorm_bwd_workspace(const NormProblem& p) {
  if (p.rows == 0) return 0;
  const Geometry g = norm_geometry(p.D, p.bf16 ? 2 : 4, true);
  return align_up((size_t)norm_grid(p, g) * p.D * sizeof(float), 256);
}

cudaError_t gated_rmsnorm_fwd(const NormProblem& p, cudaStream_t s) {
  return p.bf16 ? norm_dispatch<__nv_bfloat16>(p, false, s) : norm_dispatch<float>(p, false, s);
}

cudaError_t gated_rmsnorm_bwd(const NormProblem& p, cudaStream_t s) {
  return p.bf16 ? norm_dispatch<__nv_bfloat16>(p, true, s) : norm_dispatch<float>(p, true, s);
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
