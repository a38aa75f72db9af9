// Tensor-core (tcgen05 / TMEM / TMA) kernels for the KDA mixer, whose forget
// gate has one value per key dimension: bf16 inputs, dk = dv = 128, chunk
// C = 64, fp32 state and accumulation.
//
// Per chunk, gamma[r][d] is the within-chunk cumulative log gate of key
// dimension d, and the decay between tokens j <= r is Gam[r][j][d] =
// exp(gamma[r][d] - gamma[j][d]): it depends on d, the index the products
// sum over, so it cannot be applied to a product's output as the scalar
// gate's decay is.  It factorises instead around a per-dimension reference
// lam[d] (the middle of the chunk's gamma range in that dimension):
//   Gam[r][j][d] = Ep[r][d] Em[j][d],  Ep = exp(gamma - lam), Em = exp(lam - gamma),
// so that with the element-scaled tiles Kp = K o Ep, Km = K o Em, Qp = Q o Ep
//   A = beta_r strict_lower(Kp Km^T),   P = lower(Qp Km^T)
// are plain products.  Each factor is at most exp(range / 2); a chunk whose
// range exceeds kKdaRange in some dimension is not taken by these kernels
// (see below).  The state is kept in the chunk's reference frame,
// Ht = diag(exp(lam)) H (in TMEM as G~ = Ht^T, dv x dk), where
//   K o E H = Kp Ht,  Q o E H = Qp Ht,  E = exp(gamma),
//   H_out = diag(cf) (Ht + Km^T U),  cf = exp(gamma_last - lam),
// and one per-column pass (by cf and the next chunk's exp(lam)) moves the
// state from one chunk's frame to the next.  With W~ = T diag(beta) Kp and
// T = (I + A)^-1 the forward is the GDN chunk form with these tiles:
//   U = T diag(beta) V - W~ Ht,   O = Qp Ht + P U,   Ht' = diag(cf lam'_e)(Ht + Km^T U).
//
// Kernels:
//   prep      one CTA per chunk, every chunk at once: gamma, lam, the scaled
//             tiles, A on tcgen05 and the blocked triangular solve; writes a
//             per-chunk block (Kp|Qp, Km, T, factor vectors) to the
//             workspace, and flags the sequence when a range is too wide.
//   forward   one CTA per sequence, warp-specialised like the GDN forward,
//             loading each chunk's block with bulk copies.
//   backward  the reverse chunk scan (described at its kernel).
//
// Range limit and fallback.  The factor tiles are bf16; the backward's
// products lose precision as the per-dimension range grows (dbeta first).
// Sequences with a chunk whose range exceeds kKdaRange in some dimension
// (an average decay faster than exp(-1.25) per token across the chunk) are
// skipped by these kernels and computed exactly by the CUDA-core kernels,
// which the host launches for the flagged sequences only.

#include <algorithm>

#include "gdn.h"
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"
#include "tc_common.cuh"

namespace gdn {

cudaError_t kda_read_and_clear_status(int* status) { return tc::read_and_clear_file_status(status); }

namespace {

using namespace tc;

constexpr float kKdaRange = 80.f;

// Per-chunk block in the workspace (written by the prep kernel):
constexpr int kKT_KQ = 0;        // [Kp d0-63 | Qp d0-63 | Kp d64-127 | Qp d64-127], 8 KB each
constexpr int kKT_KM = 32768;    // [Km d0-63 | Km d64-127]
constexpr int kKT_T = 49152;     // T = (I + A)^-1, bf16 [r][j]
constexpr int kKT_VEC = 57344;   // fp32: lam[128], exp(lam)[128], cf[128], beta[64]
constexpr int kVecBytes = 1792;
constexpr int kKTBytes = kKT_VEC + kVecBytes;  // 59136 (a multiple of 128)
constexpr int kVecLam = 0, kVecElam = 128, kVecCf = 256, kVecBeta = 384;

// ---------------------------------------------------------------- prep kernel

constexpr int PT = 256;
constexpr int kP_KQ = 0;                        // K|Q tiles from TMA, scaled in place to Kp|Qp
constexpr int kP_KM = 32768;                    // Km
constexpr int kP_VEC = 49152;                   // factor vectors of this chunk
constexpr int kP_A = kP_VEC + kVecBytes;        // A fp32 [64][kLdF]
constexpr int kP_T = kP_A + 64 * kLdF * 4;      // T fp32 [64][kLdF]
constexpr int kP_S = kP_T + 64 * kLdF * 4;      // solve scratch
constexpr int kP_X = kP_S + kSolveScratch * 4;  // exchange: totals, minima, maxima of the row halves
constexpr int kP_BAR = kP_X + 3 * 256 * 4;
constexpr int kPrepSmemBytes = kP_BAR + 64 + 1024;
static_assert(2 * (kPrepSmemBytes + 1024) <= 228 * 1024, "two prep CTAs per SM");
static_assert(kP_S - kP_A >= 64 * 128 * 4, "the fp32 gate tile fits in the A and T slots");

struct KdaPrepParams {
  const float* g;         // [B, T, H, dk] (bf16 when g16)
  const float* beta;      // [B, T, H]
  unsigned char* ktiles;  // [B*H][N][kKTBytes]
  int* skip;              // [sequences * H] flags, zero before the launch
  int B, T, H, N;
  Seqs sq;
  int nseq;
  bool g16;
};

template <bool Packed, bool G16>
__global__ void __launch_bounds__(PT)
kda_tc_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                   const __grid_constant__ CUtensorMap tm_g, KdaPrepParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  int sqi, h, ci, b, tb, len, nch;
  if (!p.sq.chunk_of(blockIdx.x, p.nseq, sqi, h, ci)) return;  // past the last packed chunk
  p.sq.get_t<Packed>(sqi, b, tb, len, nch);
  const int bh = sqi * p.H + h;
  const int t0 = tb + ci * C, n = min(C, len - ci * C);
  float* vec = reinterpret_cast<float*>(sm + kP_VEC);
  float* Am = reinterpret_cast<float*>(sm + kP_A);
  float* Tm = reinterpret_cast<float*>(sm + kP_T);
  float* Sm = reinterpret_cast<float*>(sm + kP_S);
  float* xs = reinterpret_cast<float*>(sm + kP_X);  // [0,256) totals, [256,512) minima, [512,768) maxima
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + kP_BAR);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);

  grid_dep_wait();  // the previous kernel's results (and its reads of what this one writes)
  grid_dep_launch();
  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar_ld, 32768 + 64 * D * (G16 ? 2 : 4));
    tma_load_4d(sm + kP_KQ + 0, &tm_k, bar_ld, 0, h, t0, b);
    tma_load_4d(sm + kP_KQ + 8192, &tm_q, bar_ld, 0, h, t0, b);
    tma_load_4d(sm + kP_KQ + 16384, &tm_k, bar_ld, 64, h, t0, b);
    tma_load_4d(sm + kP_KQ + 24576, &tm_q, bar_ld, 64, h, t0, b);
    // the chunk's gate tile [64 tokens][128 dims] (16 KB bf16 / 32 KB fp32) into the
    // A and T slots, free until the A product, long after the gates are read
    tma_load_4d(sm + kP_A, &tm_g, bar_ld, 0, h, t0, b);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  // gamma: this thread's key dimension d and row half rh (rows 32 rh + [0, 32))
  const int d = tid & 127, rh = tid >> 7;
  float gm[32];
  {
    float mn = 0.f, mx = 0.f;
    __syncthreads();  // the barrier is initialised (thread 0, above) before anyone polls it
    __syncthreads_and(mbar_wait(bar_ld, 0));  // (a failed wait is reported below)
    if (G16) {
      const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(sm + kP_A) + d;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rh + i;
        gm[i] = r < n ? __bfloat162float(src[r * D]) : 0.f;
      }
    } else {
      const float* src = reinterpret_cast<const float*>(sm + kP_A) + d;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int r = 32 * rh + i;
        gm[i] = r < n ? src[r * D] : 0.f;
      }
    }
#pragma unroll
    for (int i = 1; i < 32; ++i) gm[i] += gm[i - 1];
    mn = gm[0];
    mx = gm[0];
#pragma unroll
    for (int i = 1; i < 32; ++i) mn = fminf(mn, gm[i]), mx = fmaxf(mx, gm[i]);
    xs[rh * 128 + d] = gm[31];
    xs[256 + rh * 128 + d] = mn;
    xs[512 + rh * 128 + d] = mx;
  }
  if (tid < 64) {
    const size_t o = ((size_t)b * p.T + t0 + tid) * p.H + h;
    vec[kVecBeta + tid] = tid < n ? p.beta[o] : 0.f;
  }
  cta_sync();
  const uint32_t tmem = *tmem_slot;
  float lam;
  {
    const float tot0 = xs[d];
    if (rh == 1) {
#pragma unroll
      for (int i = 0; i < 32; ++i) gm[i] += tot0;
    }
    const float lo = fminf(xs[256 + d], tot0 + xs[384 + d]);
    const float hi = fmaxf(xs[512 + d], tot0 + xs[640 + d]);
    lam = 0.5f * (lo + hi);
    if (!(hi - lo <= kKdaRange)) p.skip[bh] = 1;  // also catches a non-finite gate
    if (rh == 0) {
      vec[kVecLam + d] = lam;
      vec[kVecElam + d] = __expf(lam);
    } else {
      vec[kVecCf + d] = __expf(gm[31] - lam);
    }
  }
  bool ok = __syncthreads_and(mbar_wait(bar_ld, 0));
  if (ok) {
    // Kp = K o Ep, Qp = Q o Ep in place, Km = K o Em
    unsigned char* kq = sm + kP_KQ + (d >> 6) * 16384;
    unsigned char* km = sm + kP_KM + (d >> 6) * 8192;
    const int c16 = (d & 63) >> 3, e2 = (d & 7) * 2;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int r = 32 * rh + i;
      const float ep = __expf(gm[i] - lam), em = __expf(lam - gm[i]);
      const int off = sw_row_off(r, c16) + e2;
      __nv_bfloat16* kp = reinterpret_cast<__nv_bfloat16*>(kq + off);
      __nv_bfloat16* qp = reinterpret_cast<__nv_bfloat16*>(kq + 8192 + off);
      const float kv = __bfloat162float(*kp), qv = __bfloat162float(*qp);
      *kp = __float2bfloat16_rn(kv * ep);
      *qp = __float2bfloat16_rn(qv * ep);
      *reinterpret_cast<__nv_bfloat16*>(km + off) = __float2bfloat16_rn(kv * em);
    }
  }
  fence_async_shared();
  ok = __syncthreads_and(ok);
  unsigned char* dst = p.ktiles + rec_bh<Packed>(p.sq, p.N, bh, sqi, h, ci) * kKTBytes;
  if (ok && tid == 0) {
    bulk_store(dst + kKT_KQ, sm + kP_KQ, 32768);
    bulk_store(dst + kKT_KM, sm + kP_KM, 16384);
    bulk_store(dst + kKT_VEC, sm + kP_VEC, kVecBytes);
    bulk_commit_group();
    // K K^T with the decays folded in: Kp Km^T (M = 64: row r in TMEM lane 32 (r / 16) + r % 16)
    tc_fence_after();
    const uint32_t id = idesc_bf16(64, 64, false, false);
    const uint64_t dK0 = sw128_desc(smem_u32(sm), 16, 1024);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
      mma_bf16(tmem, desc_at(dK0, kP_KQ + (ks / 4) * 16384 + (ks % 4) * 32),
               desc_at(dK0, kP_KM + (ks / 4) * 8192 + (ks % 4) * 32), id, ks > 0);
    mma_commit(bar_mma);
  }
  const bool loaded = ok;
  if (ok) {
    ok = __syncthreads_and(mbar_wait(bar_mma, 0));
    tc_fence_after();
  }
  if (ok) {
    // A rows 16 quad + lane (lanes 0-15), columns 32 half + [0, 32)
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + half * 32, v);
    if (lane < 16) {
      const int r = quad * 16 + lane;
      const float br = vec[kVecBeta + r];
#pragma unroll
      for (int i = 0; i < 32; i += 4) {
        float4 a;
        const int j = half * 32 + i;
        a.x = j < r ? br * v[i] : 0.f;
        a.y = j + 1 < r ? br * v[i + 1] : 0.f;
        a.z = j + 2 < r ? br * v[i + 2] : 0.f;
        a.w = j + 3 < r ? br * v[i + 3] : 0.f;
        *reinterpret_cast<float4*>(Am + r * kLdF + j) = a;
      }
    }
    __syncthreads();
    solve_unit_lower(Am, Tm, Sm, tid, PT, [] { __syncthreads(); });
    // T as a bf16 tile in MMA-operand layout: row r = tid / 4, 16-byte chunks 2 (tid % 4) + {0, 1}
    const int r = tid >> 2;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int c8 = (tid & 3) * 2 + k;
      uint4 pk;
      uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int j = c8 * 8 + 2 * i;
        const float x0 = j <= r ? Tm[r * kLdF + j] : 0.f;
        const float x1 = j + 1 <= r ? Tm[r * kLdF + j + 1] : 0.f;
        __nv_bfloat162 b2 = __floats2bfloat162_rn(x0, x1);
        w[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(dst + kKT_T + sw_row_off(r, c8)) = pk;
    }
  } else if (tid == 0) {
    report_timeout();
    // nothing may still be writing this CTA's shared memory or TMEM at exit (bounded)
    if (!loaded) mbar_wait(bar_ld, 0, 10000);
    else mbar_wait(bar_mma, 0, 10000);
  }
  if (tid == 0) bulk_wait_all();  // the block's bulk stores have read their sources
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------- forward kernel
//
// As the GDN forward (warps 8-15 prepare chunk c+1 while warps 0-7 run the
// state chain of chunk c), with the per-chunk block of the prep kernel in
// place of the K|Q tiles and the gates:
//   preparation  T'' = T diag(beta); MMA1 [Kp;Qp] Km^T -> P = lower(Qp Km^T);
//                MMA2 W~^T = Kp^T T''^T; MMA3a U^T = V^T T''^T
//   chain        MMA3b U^T -= G~ W~^T; MMA4 O = Qp G~^T + P U;
//                MMA5 G~ += U^T Km; G~ <- G~ diag(cf lam'_e) for the next chunk.

constexpr int FT = 512;
constexpr int kF_KQ = 0;                       // 2 x 32 KB [Kp|Qp] stages
constexpr int kF_KM = 65536;                   // 2 x 16 KB Km
constexpr int kF_V = 98304;                    // 16 KB
constexpr int kF_G = 114688;                   // G~ bf16, K-major [c][d], 2 x 16 KB
constexpr int kF_W = 147456;                   // W~, MN-major rows d, 64 r
constexpr int kF_P = 163840;                   // 2 x P [r][j]
constexpr int kF_T0 = 180224;                  // T'' = T diag(beta)
constexpr int kF_U = 188416;                   // U^T [c][j] K-major
constexpr int kF_TR = 204800;                  // 2 x T from the prep kernel
constexpr int kF_VEC = 221184;                 // 2 x factor vectors
constexpr int kF_CF = kF_VEC + 2 * kVecBytes;  // chain's copy of the current chunk's cf
constexpr int kF_BAR = kF_CF + 512;
constexpr int kFwdSmemBytes = kF_BAR + 128 + 1024;
static_assert(kFwdSmemBytes <= 227 * 1024, "shared memory budget");

constexpr uint32_t kTmKQ = 0, kTmW = 64, kTmU0 = 128, kTmO = 256, kTmG = 384, kTmCols = 512;

struct KdaFwdParams {
  const float* h0;
  __nv_bfloat16* o;
  float* ht;
  __nv_bfloat16* states;        // optional: bf16 G~ tile of every chunk's entry state
  const unsigned char* ktiles;  // the prep kernel's per-chunk blocks
  const int* skip;              // sequences the CUDA-core kernels take
  int B, T, H, N;
  Seqs sq;
};

template <bool Packed>
__global__ void __launch_bounds__(FT, 1)
kda_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  KdaFwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, half = (warp >> 2) & 1, grp = warp >> 3;
  const int row = quad * 32 + lane;
  const int bh = blockIdx.x, sqi = bh / p.H, h = bh % p.H;
  int b = 0, tb = 0, slen = 0, NL = 0;  // batch row, first token, length, chunks (after the wait)

  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + kF_BAR);  // [2] stage loaded
  uint64_t* bar_v = bar_kq + 2;
  uint64_t* bar_p = bar_kq + 3;
  uint64_t* bar_s = bar_kq + 4;
  uint64_t* bar_pd = bar_kq + 5;
  uint64_t* bar_wf = bar_kq + 6;
  uint64_t* bar_p1 = bar_kq + 7;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_kq + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* cnt = reinterpret_cast<int*>(tmem_slot + 2);  // [0..1] kq issued, [2..3] kq waited, [4] v issued, [5] v waited, [6] early MMA1
  float* cf = reinterpret_cast<float*>(sm + kF_CF);

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&bar_kq[i], 1);
    *abort_flag = 0;
    for (int i = 0; i < 7; ++i) cnt[i] = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmCols);
    tmem_relinquish();
  }
  cta_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
  // operand descriptors: every tile's is a base descriptor plus its offset
  const uint64_t dK0 = sw128_desc(smem_u32(sm), 16, 1024);     // K-major tiles
  const uint64_t dM0 = sw128_desc(smem_u32(sm), 16384, 1024);  // MN-major, halves 16 KB apart
  const uint64_t dV0 = sw128_desc(smem_u32(sm), 8192, 1024);   // MN-major, halves 8 KB apart
  grid_dep_wait();
  grid_dep_launch();
  p.sq.get_t<Packed>(sqi, b, tb, slen, NL);
  if (p.skip[bh] || (Packed && NL == 0)) {  // the CUDA-core kernels take it (or it is empty)
    if (!p.skip[bh] && p.ht)      // an empty packed sequence keeps its initial state
      for (int i = tid; i < D * D; i += FT) p.ht[(size_t)bh * D * D + i] = p.h0 ? p.h0[(size_t)bh * D * D + i] : 0.f;
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmCols);
    return;
  }

  auto blk = [&](int ci) { return p.ktiles + rec_bh<Packed>(p.sq, p.N, bh, sqi, h, ci) * kKTBytes; };
  auto vec = [&](int ci) { return reinterpret_cast<const float*>(sm + kF_VEC + (ci & 1) * kVecBytes); };
  auto load_kq = [&](int ci) {
    const int st = ci & 1;
    const unsigned char* src = blk(ci);
    mbar_arrive_expect_tx(&bar_kq[st], kKTBytes);
    bulk_load(sm + kF_KQ + st * 32768, src + kKT_KQ, 32768, &bar_kq[st]);
    bulk_load(sm + kF_KM + st * 16384, src + kKT_KM, 16384, &bar_kq[st]);
    bulk_load(sm + kF_TR + st * 8192, src + kKT_T, 8192, &bar_kq[st]);
    bulk_load(sm + kF_VEC + st * kVecBytes, src + kKT_VEC, kVecBytes, &bar_kq[st]);
    cnt[st] += 1;
  };
  auto load_v = [&](int ci) {
    mbar_arrive_expect_tx(bar_v, 16384);
    const int t0 = tb + ci * C;
    tma_load_4d(sm + kF_V, &tm_v, bar_v, 0, h, t0, b);
    tma_load_4d(sm + kF_V + 8192, &tm_v, bar_v, 64, h, t0, b);
    cnt[4] += 1;
  };
  auto state_dst = [&](int ci) -> unsigned char* {
    return p.states ? reinterpret_cast<unsigned char*>(p.states) + rec_bh<Packed>(p.sq, p.N, bh, sqi, h, ci) * (size_t)32768
                    : nullptr;
  };
  const bool want_o = p.o != nullptr;

  if (tid == 0) {
    load_kq(0);
    if (NL > 1) load_kq(1);
    load_v(0);
  }
  bool ok = true;

  if (grp == 0) {
    // ============================== chain group ==============================
    const int gt = tid;
    // initial state in chunk 0's frame: G~ = h0^T diag(exp(lam_0)) (fp32 in TMEM, bf16 tile)
    ok = group_and(kBarChain, kGroup, mbar_wait(&bar_kq[0], 0));
    if (ok) {
      const float* el = vec(0) + kVecElam;
      float v[32];
#pragma unroll
      for (int q32 = 0; q32 < 2; ++q32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int d = half * 64 + q32 * 32 + i;
          v[i] = p.h0 ? p.h0[((size_t)bh * D + d) * D + row] * el[d] : 0.f;
        }
        tmem_st32(tmem + lane_base + kTmG + half * 64 + q32 * 32, v);
        store_chunks(sm + kF_G + half * 16384, row, q32 * 4, v, 4);
      }
      fence_async_shared();
      group_sync_tc(kBarChain);
      if (gt == 0 && p.states) {
        bulk_store(state_dst(0), sm + kF_G, 32768);
        bulk_commit_group();
      }
    }
    uint32_t s_phase = 0;
    for (int ci = 0; ci < NL && ok; ++ci) {
      const int s = ci & 1, t0 = tb + ci * C, nrow = min(C, slen - ci * C);
      ok = group_and(kBarChain, kGroup, mbar_wait(bar_pd, ci & 1) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      {
        // W~^T (TMEM) -> W~ tile, MN-major: row d holds W~[0..63][d]
        float w[32];
        tmem_ld32(tmem + lane_base + kTmW + half * 32, w);
        store_chunks(sm + kF_W, row, half * 4, w, 4);
      }
      if (gt < 128) cf[gt] = vec(ci)[kVecCf + gt];  // kept past the stage's reload
      fence_async_shared();
      group_sync_tc(kBarChain);
      if (gt == 0) mbar_arrive(bar_wf);
      const uint32_t st_kq = smem_u32(sm + kF_KQ + s * 32768);
      const uint32_t st_km = smem_u32(sm + kF_KM + s * 16384);
      const uint32_t tmU = kTmU0 + 64 * s;
      if (gt == 0) {
        // MMA3b: U^T += -G~ W~^T
        const uint32_t id3 = idesc_bf16(128, 64, false, true, true);
        #pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_bf16(tmem + tmU, desc_at(dK0, kF_G + (ks / 4) * 16384 + (ks % 4) * 32),
                   desc_at(dM0, kF_W + ks * 2048), id3, 1);
        // MMA4a: O = Qp G~^T  (M = 64: A = Qp rows r; B = G~ tile rows c)
        const uint32_t id4 = idesc_bf16(64, 128, false, false);
        for (int ks = 0; ks < (want_o ? 8 : 0); ++ks) {
          const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
          mma_bf16(tmem + kTmO, desc_at(dK0, (kF_KQ + s * 32768) + 8192 + off),
                   desc_at(dK0, kF_G + off), id4, ks > 0);
        }
        mma_commit(bar_s);
        bulk_wait_read_all();  // the last output rows staged in the U^T slot have been read
      }
      ok = group_and(kBarChain, kGroup, mbar_wait(bar_s, s_phase));
      s_phase ^= 1;
      tc_fence_after();
      if (!ok) break;
      {
        float u[32];
        tmem_ld32(tmem + lane_base + tmU + half * 32, u);
        store_chunks(sm + kF_U, row, half * 4, u, 4);
      }
      fence_async_shared();
      group_sync_tc(kBarChain);
      if (gt == 0) {
        // MMA4b: O += P U
        const uint32_t id4 = idesc_bf16(64, 128, false, false);
        #pragma unroll
        for (int ks = 0; ks < (want_o ? 4 : 0); ++ks)
          mma_bf16(tmem + kTmO, desc_at(dK0, kF_P + s * 8192 + ks * 32),
                   desc_at(dK0, kF_U + ks * 32), id4, 1);
        // MMA5: G~ += U^T Km  (B: Km tile, MN-major N = d, K = j)
        const uint32_t id5 = idesc_bf16(128, 128, false, true);
        #pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTmG, desc_at(dK0, kF_U + ks * 32),
                   desc_at(dV0, (kF_KM + s * 16384) + ks * 2048), id5, 1);
        mma_commit(bar_s);
        bulk_wait_read_all();  // the last entry-state copy has read the tile rewritten next
      }
      ok = group_and(kBarChain, kGroup, mbar_wait(bar_s, s_phase));
      s_phase ^= 1;
      tc_fence_after();
      if (!ok) break;
      if (gt == 0 && ci + 2 < NL) load_kq(ci + 2);  // this stage is no longer read
      if (want_o) {
        const int r = quad * 16 + lane;
#pragma unroll
        for (int q32 = 0; q32 < 2; ++q32) {
          float v[32];
          tmem_ld32(tmem + lane_base + kTmO + half * 64 + q32 * 32, v);
          if (lane < 16) store_chunks(sm + kF_U + half * 8192, r, q32 * 4, v, 4);
        }
      }
      {
        // the state at the chunk's end, moved into the next chunk's frame
        // (diag(cf exp(lam'))); after the last chunk, into the true frame (cf)
        const bool more = ci + 1 < NL;
        if (more) {
          // the next chunk's block holds exp(lam'); its stage was requested a chunk ago
          ok = group_and(kBarChain, kGroup, mbar_wait(&bar_kq[(ci + 1) & 1], ((ci + 1) >> 1) & 1));
          if (!ok) break;
        }
        const float* el = vec(ci + 1) + kVecElam;
        unsigned char* dstate = more ? state_dst(ci + 1) : nullptr;
        float v[32];
#pragma unroll
        for (int q32 = 0; q32 < 2; ++q32) {
          const uint32_t ta = tmem + lane_base + kTmG + half * 64 + q32 * 32;
          tmem_ld32(ta, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int d = half * 64 + q32 * 32 + i;
            v[i] *= more ? cf[d] * el[d] : cf[d];
          }
          tmem_st32(ta, v);
          if (more) store_chunks(sm + kF_G + half * 16384, row, q32 * 4, v, 4);
        }
        fence_async_shared();
        group_sync_tc(kBarChain);
        // the output rows: a tensor store, or row by row for a packed
        // sequence's partial last chunk (the rows past it belong to the next)
        const bool rowwise = Packed && want_o && nrow < C;
        if (rowwise)
          store_rows_bf16(sm + kF_U, p.o + (((size_t)b * p.T + t0) * p.H + h) * D, (size_t)p.H * D, nrow,
                          gt, kGroup);
        if (gt == 0 && (dstate || want_o)) {
          if (dstate) bulk_store(dstate, sm + kF_G, 32768);
          if (want_o && !rowwise) {
            tma_store_4d(&tm_o, sm + kF_U, 0, h, t0, b);
            tma_store_4d(&tm_o, sm + kF_U + 8192, 64, h, t0, b);
          }
          bulk_commit_group();
        }
      }
    }
    if (gt == 0) bulk_wait_all();
    if (!ok) *abort_flag = 1;
    if (ok && p.ht) {
      float v[32];
#pragma unroll
      for (int q32 = 0; q32 < 2; ++q32) {
        tmem_ld32(tmem + lane_base + kTmG + half * 64 + q32 * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) p.ht[((size_t)bh * D + half * 64 + q32 * 32 + i) * D + row] = v[i];
      }
    }
  } else {
    // =========================== preparation group ===========================
    const int pt = tid - kGroup;
    auto psync = [&]() { group_sync(kBarPrep, kGroup); };
    volatile int* early_mma1 = cnt + 6;
    if (pt == 0) *early_mma1 = 0;
    auto issue_mma1 = [&](int cn) {
      // MMA1: [Kp;Qp] Km^T, M = 128 N = 64 K = 128 (lanes 64-127: Qp Km^T)
      const uint32_t kq = smem_u32(sm + kF_KQ + (cn & 1) * 32768);
      const uint32_t km = smem_u32(sm + kF_KM + (cn & 1) * 16384);
      const uint32_t idesc = idesc_bf16(128, 64, false, false);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kTmKQ, desc_at(dK0, (kF_KQ + (cn & 1) * 32768) + (ks / 4) * 16384 + (ks % 4) * 32),
                 desc_at(dK0, (kF_KM + (cn & 1) * 16384) + (ks / 4) * 8192 + (ks % 4) * 32), idesc, ks > 0);
      mma_commit(bar_p1);
    };
    uint32_t p_phase = 0;
    for (int ci = 0; ci < NL; ++ci) {
      const int s = ci & 1;
      const uint32_t st_kq = smem_u32(sm + kF_KQ + s * 32768);
      ok = group_and(kBarPrep, kGroup, mbar_wait(&bar_kq[s], (ci >> 1) & 1) && !*abort_flag);
      if (!ok) break;
      if (pt == 0) cnt[2 + s] += 1;
      if (want_o && pt == 0 && !*early_mma1) issue_mma1(ci);
      {
        // T'' = T diag(beta): this thread's 16-byte column chunk c8 of rows r0 and r0 + 32
        const float* bt = vec(ci) + kVecBeta;
        const int c8 = pt & 7, r0 = pt >> 3;
        float sb[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sb[k] = bt[c8 * 8 + k];
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int off = sw_row_off(r0 + 32 * rr, c8);
          const uint4 raw = *reinterpret_cast<const uint4*>(sm + kF_TR + s * 8192 + off);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
          uint4 o0;
          uint32_t* w0 = reinterpret_cast<uint32_t*>(&o0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 t = __bfloat1622float2(h2[k]);
            __nv_bfloat162 x0 = __floats2bfloat162_rn(t.x * sb[2 * k], t.y * sb[2 * k + 1]);
            w0[k] = *reinterpret_cast<uint32_t*>(&x0);
          }
          *reinterpret_cast<uint4*>(sm + kF_T0 + off) = o0;
        }
      }
      if (want_o) {
        ok = group_and(kBarPrep, kGroup, mbar_wait(bar_p1, ci & 1));
        tc_fence_after();
        if (!ok) break;
        // P = lower(Qp Km^T) from TMEM lanes 64-127
        if (row >= 64) {
          const int r = row - 64;
          float v[32];
          if (quad == 2 && half == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          } else {
            tmem_ld32(tmem + lane_base + kTmKQ + half * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = half * 32 + i <= r ? v[i] : 0.f;
          }
          store_chunks(sm + kF_P + s * 8192, r, half * 4, v, 4);
        }
      }
      ok = group_and(kBarPrep, kGroup, mbar_wait(bar_v, ci & 1));
      if (!ok) break;
      if (pt == 0) cnt[5] += 1;
      if (ci > 0) {
        ok = group_and(kBarPrep, kGroup, mbar_wait(bar_wf, (ci - 1) & 1));
        if (!ok) break;
      }
      fence_async_shared();
      tc_fence_before();
      psync();
      tc_fence_after();
      if (pt == 0) {
        // MMA2: W~^T = Kp^T T''^T  (A: Kp MN-major, M = d; B: T'' K-major, N = r)
        const uint32_t id2 = idesc_bf16(128, 64, true, false);
        #pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTmW, desc_at(dM0, (kF_KQ + s * 32768) + ks * 2048),
                   desc_at(dK0, kF_T0 + ks * 32), id2, ks > 0);
        // MMA3a: U^T = V^T T''^T
        #pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTmU0 + 64 * s, desc_at(dV0, kF_V + ks * 2048),
                   desc_at(dK0, kF_T0 + ks * 32), id2, ks > 0);
        mma_commit(bar_p);
      }
      ok = group_and(kBarPrep, kGroup, mbar_wait(bar_p, p_phase));
      p_phase ^= 1;
      tc_fence_after();
      if (!ok) break;
      if (pt == 0 && ci + 1 < NL) load_v(ci + 1);
      if (want_o && pt == 0) {
        const int cn = ci + 1;
        *early_mma1 = (cn < NL && mbar_test_wait(&bar_kq[cn & 1], (cn >> 1) & 1)) ? 1 : 0;
        if (*early_mma1) issue_mma1(cn);
      }
      tc_fence_before();
      psync();
      if (pt == 0) mbar_arrive(bar_pd);
    }
    if (!ok) *abort_flag = 1;
  }

  __syncthreads();
  if (*abort_flag) {
    if (tid == 0) {
      report_timeout();
      for (int st = 0; st < 2; ++st)
        for (int k = cnt[2 + st]; k < cnt[st]; ++k) mbar_wait(&bar_kq[st], k & 1, 10000);
      for (int k = cnt[5]; k < cnt[4]; ++k) mbar_wait(bar_v, k & 1, 10000);
    }
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

// ---------------------------------------------------------------- backward kernel
//
// Reverse chunk scan, one CTA (512 threads) per sequence, as the GDN backward
// with the prep kernel's scaled tiles.  The state gradient is held in TMEM as
// dG (dv x dk, fp32); on entering chunk c it is dG^ = dG_out diag(cf_c), the
// gradient of the chunk's frame state, which is also its bf16 MMA operand.
// With R = V - Kp Ht, U = T diag(beta) R, dU = Km dG^ + P^T dO,
// dZ = T^T dU, dR = diag(beta) dZ, dA = -strict_lower(dZ U^T),
// dP = lower(dO U^T), M = diag(beta) dA, Po = strict_lower(dP):
//
//   MMA1  [Kp;Qp] Km^T, -G~ Kp^T, dG^ Km^T      (K K^T, Q K^T -> P, R, dU part)
//   MMA   dO^T P                                  (dU part)
//   MMA   U = beta R + (T - I) beta R,  dZ = dU + (T - I)^T dU
//         (the identity parts added in fp32, so that dbeta, which sums
//         dZ o R with much cancellation when gates decay fast, sees dZ and
//         U at fp32 rather than at the bf16 precision of the product operands)
//   MMA   [dZ; dO] U^T                            (dA, dP)
//   MMA   dG <- dG^ + dO^T Qp - dR^T Kp           (then diag(exp(lam)) in the epilogue:
//                                                  the gradient of the chunk's entry state)
//   MMA   four accumulators, transposed ([d][token]):
//           aQ = dO Ht^T + Po Km          aP = -dR Ht^T + M Km
//           aF = U dG^                    aM = Po^T Qp + M^T Kp
//
// and, with Ep and Em formed in fp32 from the chunk's gate tile,
//   dq = Ep aQ + diag(dP) K,   dk = Ep aP + Em (aF + aM) + diag(dP) Q,
//   dgamma = Qp o aQ + Kp o aP - Km o (aF + aM),
//   dg = reverse cumsum of dgamma in the chunk + sum_c dG^ o G~ + colsum(Km o aF).
// dgamma holds no product with its own token's Q and K (the diagonal of dP
// enters dq and dk separately, and would cancel exactly in dgamma), and it
// needs no per-element exponential: the scaled tiles carry the decays.

constexpr int BT = 512;
constexpr int kB_KQ = 0;                      // [Kp|Qp]
constexpr int kB_KM = 32768;                  // Km
constexpr int kB_ZO = 49152;                  // [dZ h0 | dO h0 | dZ h1 | dO h1]; g (d 64-127) in the dZ halves at the end
constexpr int kB_GI = 81920;                  // G~ of the chunk's entry
constexpr int kB_DG = 114688;                 // dG^ bf16
constexpr int kB_V = 147456;                  // V; g (d 0-63) at the end
constexpr int kB_T = kB_V + 16384;            // T (diagonal zeroed); then dv staging with P; then M
constexpr int kB_P = kB_T + 8192;             // P; then Po
constexpr int kB_X = kB_P + 8192;             // X0: beta R^T, then U^T, then dq staging; X1: dU^T, then dR^T, then dk staging
constexpr int kB_VEC = kB_X + 2 * 16384;      // 2 x factor vectors
constexpr int kB_RED = kB_VEC + 2 * kVecBytes;  // 1536 floats of reduction scratch
constexpr int kB_SM = kB_RED + 1536 * 4;        // db1[64] db2[64] dPd[64] carry1[128]
constexpr int kB_BAR = kB_SM + 320 * 4;
constexpr int kBwdSmemBytes = kB_BAR + 128 + 1024;
static_assert(kBwdSmemBytes <= 227 * 1024, "shared memory budget");
// reduction scratch regions
constexpr int kR_SUM = 0;     // cta_sum_rows16 scratch (256)
constexpr int kR_DB2 = 256;   // dbeta part 2 partials [cg][r] (256)
constexpr int kR_COL = 512;   // carry1 partials [quad][d] (512); then dgamma totals [cg][d]
constexpr int kR_TOT = 0;     // gamma totals [cg][d] (last epilogue)
constexpr int kR_C2 = 1024;   // carry2 partials [cg][d] (last epilogue)

constexpr uint32_t kBtKQ = 0, kBtR = 64, kBtX1 = 128, kBtX2 = 192, kBtU = 256, kBtZ = 320, kBtG = 384;
constexpr uint32_t kBtAQ = 0, kBtAP = 64, kBtAF = 128, kBtAM = 192;  // after the dA / dP epilogue

struct KdaBwdParams {
  const float* dht;
  const unsigned char* ktiles;   // the prep kernel's per-chunk blocks
  const unsigned char* states;   // [B*H][N][32 KB] bf16 G~ tiles
  const int* skip;
  float* dbeta;
  float* dh0;
  __nv_bfloat16* dq;   // the token gradients, for the row-by-row stores of a
  __nv_bfloat16* dk;   // packed sequence's partial last chunk
  __nv_bfloat16* dv;
  float* dg;
  int B, T, H, N;
  Seqs sq;
};

// Each thread holds v[i], i < 32, for tile column 32 cg + i of its TMEM lane;
// lane l of the warp ends with the sum of column 32 cg + l over the warp's 32
// lanes (31 exchanges), stored to red[quad * 128 + 32 cg + l].
__device__ __forceinline__ void warp_colsum32(float (&v)[32], float* red, int quad, int cg, int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int off = 16 >> step;
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      if (i < off) {
        const float send = up ? v[i] : v[i + off];
        const float keep = up ? v[i + off] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
  }
  red[quad * 128 + cg * 32 + lane] = v[0];
}

// fp32 gate tile element (token r, key dimension d) as loaded by four TMA
// boxes of 32 dimensions: d 0-63 in the V slot, d 64-127 in the dZ halves
__device__ __forceinline__ float* gate_elem(unsigned char* sm, int r, int d) {
  const int blk = d >> 5;
  unsigned char* base = blk < 2 ? sm + kB_V + blk * 8192 : sm + kB_ZO + (blk - 2) * 16384;
  return reinterpret_cast<float*>(base + r * 128 + (d & 31) * 4);
}

// bf16 gate tile element as loaded by two TMA boxes of 64 dimensions: d 0-63
// at the start of the V slot, d 64-127 at the start of the dZ halves (both
// inside the fp32 tile's footprint, which the in-place dg sums reuse once
// every thread has read its gate values)
__device__ __forceinline__ float gate_elem16(const unsigned char* sm, int r, int d) {
  const unsigned char* base = d < 64 ? sm + kB_V : sm + kB_ZO;
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(base + r * 128 + (d & 63) * 2));
}

template <bool Packed, bool G16>
__global__ void __launch_bounds__(BT, 1)
kda_tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_dq,
                  const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                  const __grid_constant__ CUtensorMap tm_dg, KdaBwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, cg = warp >> 2;
  const int row = quad * 32 + lane;
  const int bh = blockIdx.x, sqi = bh / p.H, h = bh % p.H;
  int b = 0, tb = 0, slen = 0, NN = 0;  // batch row, first token, length, chunks (after the wait)

  float* red = reinterpret_cast<float*>(sm + kB_RED);
  float* db1 = reinterpret_cast<float*>(sm + kB_SM);
  float* db2 = db1 + 64;
  float* dPd = db2 + 64;
  float* carry1 = dPd + 64;
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + kB_BAR);
  uint64_t* bar_mma = bar_load + 1;
  uint64_t* bar_v = bar_load + 2;
  uint64_t* bar_vec = bar_load + 3;
  uint64_t* bar_g = bar_load + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_load + 5);
  const uint32_t sKQ = smem_u32(sm + kB_KQ), sKM = smem_u32(sm + kB_KM), sZO = smem_u32(sm + kB_ZO);
  const uint32_t sGI = smem_u32(sm + kB_GI), sDG = smem_u32(sm + kB_DG);
  const uint32_t sT = smem_u32(sm + kB_T), sP = smem_u32(sm + kB_P);
  const uint32_t sX0 = smem_u32(sm + kB_X), sX1 = sX0 + 16384;

  if (tid == 0) {
    for (int i = 0; i < 5; ++i) mbar_init(&bar_load[i], 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
    tma_prefetch_desc(&tm_g);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmCols);
    tmem_relinquish();
  }
  cta_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lb = (uint32_t)(quad * 32) << 16;
  grid_dep_wait();
  grid_dep_launch();
  if constexpr (Packed) p.sq.get_t<true>(sqi, b, tb, slen, NN);
  else b = sqi, slen = p.T, NN = p.N;
  if (p.skip[bh]) {  // this sequence is computed by the CUDA-core kernels
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmCols);
    return;
  }
  if (Packed && NN == 0) {  // an empty packed sequence: the state gradient passes through
    if (p.dh0)
      for (int i = tid; i < D * D; i += BT) p.dh0[(size_t)bh * D * D + i] = p.dht ? p.dht[(size_t)bh * D * D + i] : 0.f;
    cta_sync();
    if (warp == 0) tmem_dealloc(tmem, kTmCols);
    return;
  }

  auto blk = [&](int ci) { return p.ktiles + (Packed ? p.sq.template rec_t<true>(sqi, h, ci) : (size_t)bh * p.N + ci) * kKTBytes; };
  auto vec = [&](int ci) { return reinterpret_cast<const float*>(sm + kB_VEC + (ci & 1) * kVecBytes); };
  // loads (thread 0): the main tiles of chunk cn on bar_load, announced in full
  // with the first part (G~, T, dO) and completed by the second (Kp|Qp, Km)
  constexpr uint32_t kMainBytes = 32768 + 16384 + 8192 + 32768 + 16384;
  int inflight = -1, parts = 0;
  auto issue_main1 = [&](int cn) {
    inflight = cn;
    parts = 1;
    mbar_arrive_expect_tx(bar_load, kMainBytes);
    bulk_load(sm + kB_GI, p.states + (Packed ? p.sq.template rec_t<true>(sqi, h, cn) : (size_t)bh * p.N + cn) * 32768, 32768, bar_load);
    bulk_load(sm + kB_T, blk(cn) + kKT_T, 8192, bar_load);
    tma_load_4d(sm + kB_ZO + 8192, &tm_do, bar_load, 0, h, tb + cn * C, b);
    tma_load_4d(sm + kB_ZO + 24576, &tm_do, bar_load, 64, h, tb + cn * C, b);
  };
  auto issue_main2 = [&](int cn) {
    parts = 2;
    bulk_load(sm + kB_KQ, blk(cn) + kKT_KQ, 32768, bar_load);
    bulk_load(sm + kB_KM, blk(cn) + kKT_KM, 16384, bar_load);
  };
  int v_issued = 0, v_waited = 0, vec_issued = 0, vec_waited = 0, g_issued = 0, g_waited = 0;
  auto issue_v = [&](int cn) {
    mbar_arrive_expect_tx(bar_v, 16384);
    tma_load_4d(sm + kB_V, &tm_v, bar_v, 0, h, tb + cn * C, b);
    tma_load_4d(sm + kB_V + 8192, &tm_v, bar_v, 64, h, tb + cn * C, b);
    ++v_issued;
  };
  auto issue_vec = [&](int cn) {
    mbar_arrive_expect_tx(bar_vec, kVecBytes);
    bulk_load(sm + kB_VEC + (cn & 1) * kVecBytes, blk(cn) + kKT_VEC, kVecBytes, bar_vec);
    ++vec_issued;
  };

  bool ok = true;
  if (tid == 0) {
    issue_vec(NN - 1);
    issue_main1(NN - 1);
    issue_main2(NN - 1);
    issue_v(NN - 1);
  }
  // dG^ of the last chunk: dht diag(cf)  (fp32 in TMEM, bf16 tile)
  const int g_region = cg >> 1, g_chunk0 = (cg & 1) * 4;
  const uint32_t t_dg = tmem + lb + kBtG + cg * 32;
  auto write_dg = [&](const float (&g)[32]) {
    unsigned char* tile = sm + kB_DG + g_region * 16384;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint4 pk;
      uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(g[k * 8 + 2 * i], g[k * 8 + 2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(tile + sw_row_off(row, g_chunk0 + k)) = pk;
    }
  };
  ok = __syncthreads_and(mbar_wait(bar_vec, 0));
  vec_waited = 1;
  if (ok) {
    const float* cfv = vec(NN - 1) + kVecCf;
    float g[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int d = cg * 32 + i;
      g[i] = p.dht ? p.dht[((size_t)bh * D + d) * D + row] * cfv[d] : 0.f;
    }
    tmem_st32(t_dg, g);
    write_dg(g);
  }

  uint32_t mma_phase = 0, load_phase = 0;
  auto mma_wait = [&]() {
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
  };

  for (int ci = NN - 1; ci >= 0 && ok; --ci) {
    const int t0 = tb + ci * C, n = min(C, slen - ci * C);
    const bool rowwise = Packed && n < C;  // a packed sequence's partial last chunk
    const float* vc = vec(ci);
    const float* bt = vc + kVecBeta;
    fence_async_shared();  // the dG^ tile written last chunk, for MMA1 (after the barrier below)
    if (tid == 0) {
      if (ci < NN - 1) {
        bulk_wait_read_all();  // the last chunk's dg, dq, dk stores have read the V slot
        issue_v(ci);
      }
      if (ci > 0) issue_vec(ci - 1);
    }
    ok = __syncthreads_and(mbar_wait(bar_load, load_phase));
    if (!ok) break;
    load_phase ^= 1;
    inflight = -1;
    if (rowwise) {
      // rows past the sequence hold the next one's dO: zero them (their gates
      // and beta are already masked)
      for (int i = tid; i < (C - n) * 16; i += BT) {
        const int r = n + (i >> 4), hh = (i >> 3) & 1, c8 = i & 7;
        *reinterpret_cast<uint4*>(sm + kB_ZO + hh * 16384 + 8192 + r * 128 + c8 * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    // T - I: the products take the off-diagonal part, the identity is added in fp32
    if (tid < 64)
      *reinterpret_cast<__nv_bfloat16*>(sm + kB_T + sw_row_off(tid, tid >> 3) + (tid & 7) * 2) =
          __float2bfloat16_rn(0.f);
    // ---- MMA1: [Kp;Qp] Km^T;  -G~ Kp^T;  dG^ Km^T
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      const uint32_t idn = idesc_bf16(128, 64, false, false, true);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        const uint32_t offm = (ks / 4) * 8192 + (ks % 4) * 32;
        mma_bf16(tmem + kBtKQ, sw128_desc(sKQ + off, 16, 1024), sw128_desc(sKM + offm, 16, 1024), id, ks > 0);
        mma_bf16(tmem + kBtR, sw128_desc(sGI + off, 16, 1024), sw128_desc(sKQ + off, 16, 1024), idn, ks > 0);
        mma_bf16(tmem + kBtX1, sw128_desc(sDG + off, 16, 1024), sw128_desc(sKM + offm, 16, 1024), id, ks > 0);
      }
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // P = lower(Qp Km^T) from TMEM lanes 64-127
    if (row >= 64) {
      const int r = row - 64;
      float v[16];
      tmem_ld16(tmem + lb + kBtKQ + cg * 16, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = cg * 16 + i <= r ? v[i] : 0.f;
      store_chunks(sm + kB_P, r, cg * 2, v, 2);
    }
    fence_async_shared();
    cta_sync();
    // ---- dO^T P
    if (tid == 0) {
      const uint32_t idmm = idesc_bf16(128, 64, true, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtX2, sw128_desc(sZO + 8192 + ks * 2048, 16384, 1024),
                 sw128_desc(sP + ks * 2048, 16384, 1024), idmm, ks > 0);
      mma_commit(bar_mma);
      bulk_wait_read_all();  // the last chunk's dq / dk staging (X0, X1) and g / dg slots have been read
    }
    ok = __syncthreads_and(mbar_wait(bar_v, v_waited & 1));
    ++v_waited;
    if (!ok) break;
    mma_wait();
    if (!ok) break;
    // ---- E3: beta R^T -> X0, dU^T -> X1  (this thread: row c, columns j = 16 cg + i)
    {
      float a[16], x[16];
      tmem_ld16(tmem + lb + kBtR + cg * 16, a);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = cg * 16 + i;
        a[i] = bt[j] * (tile_elem(sm + kB_V + (row >> 6) * 8192, j, row & 63) + a[i]);
      }
      store_chunks(sm + kB_X, row, cg * 2, a, 2);
      tmem_ld16(tmem + lb + kBtX1 + cg * 16, a);
      tmem_ld16(tmem + lb + kBtX2 + cg * 16, x);
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] += x[i];
      store_chunks(sm + kB_X + 16384, row, cg * 2, a, 2);
    }
    fence_async_shared();
    cta_sync();
    // ---- (T - I) beta R and (T - I)^T dU
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      const uint32_t idm = idesc_bf16(128, 64, false, true);
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tmem + kBtU, sw128_desc(sX0 + ks * 32, 16, 1024), sw128_desc(sT + ks * 32, 16, 1024), id,
                 ks > 0);
        mma_bf16(tmem + kBtZ, sw128_desc(sX1 + ks * 32, 16, 1024), sw128_desc(sT + ks * 2048, 16384, 1024),
                 idm, ks > 0);
      }
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // ---- E4: carry terms, U^T -> X0, dR^T -> X1, dZ rows -> ZO, dv, dbeta part 1
    {
      {
        // sum over c of dG^ o G~ for this thread's columns d = 32 cg + i
        float g[32];
        tmem_ld32(t_dg, g);
        const unsigned char* tile = sm + kB_GI + g_region * 16384;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 pk = *reinterpret_cast<const uint4*>(tile + sw_row_off(row, g_chunk0 + k));
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f2 = __bfloat1622float2(h2[i]);
            g[k * 8 + 2 * i] *= f2.x;
            g[k * 8 + 2 * i + 1] *= f2.y;
          }
        }
        warp_colsum32(g, red + kR_COL, quad, cg, lane);
      }
      float u[16], rr[16];
      tmem_ld16(tmem + lb + kBtR + cg * 16, rr);
      tmem_ld16(tmem + lb + kBtU + cg * 16, u);
      const int hv = row >> 6, cc = row & 63;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = cg * 16 + i;
        rr[i] += tile_elem(sm + kB_V + hv * 8192, j, cc);  // R^T
        u[i] = fmaf(bt[j], rr[i], u[i]);                    // U = beta R + (T - I) beta R
      }
      store_chunks(sm + kB_X, row, cg * 2, u, 2);
      float z[16];
      tmem_ld16(tmem + lb + kBtZ + cg * 16, z);
      tmem_ld16(tmem + lb + kBtX1 + cg * 16, u);
#pragma unroll
      for (int i = 0; i < 16; ++i) z[i] += u[i];
      tmem_ld16(tmem + lb + kBtX2 + cg * 16, u);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = cg * 16 + i;
        z[i] += u[i];                                // dZ = dU + (T - I)^T dU
        rr[i] *= z[i];                               // dZ_jc R_jc
        z[i] *= bt[j];                               // dR
      }
      {
        // dv = dR (T and P are read for the last time) and the dZ rows of the
        // [dZ; dO] operand, token-major: transposed stores of this warp's block
        // (the same sum dZ = Z + X1 + X2, read again in the 16x256b layout)
        const uint32_t tz = tmem + lb + kBtZ + cg * 16, t1 = tmem + lb + kBtX1 + cg * 16,
                       t2 = tmem + lb + kBtX2 + cg * 16;
        stage_tmem_block(sm + kB_T, 8192, tz, quad * 32, cg * 16,
                         [&](int j, float zz) { return bt[j] * zz; }, t1, t2);
        stage_tmem_block(sm + kB_ZO, 16384, tz, quad * 32, cg * 16, [](int, float zz) { return zz; }, t1,
                         t2);
      }
      store_chunks(sm + kB_X + 16384, row, cg * 2, z, 2);  // dR^T
      cta_sum_rows16(rr, red + kR_SUM, db1);
    }
    fence_async_shared();
    cta_sync();
    // ---- G4: [dZ; dO] U^T  (lanes 0-63: dZ U^T, lanes 64-127: dO U^T)
    if (rowwise)
      store_rows_bf16(sm + kB_T, p.dv + (((size_t)b * p.T + t0) * p.H + h) * D, (size_t)p.H * D, n, tid,
                      BT);
    if (tid == 0) {
      if (!rowwise) {
        tma_store_4d(&tm_dv, sm + kB_T, 0, h, t0, b);
        tma_store_4d(&tm_dv, sm + kB_T + 8192, 64, h, t0, b);
      }
      bulk_commit_group();
      // the gate tile, d 0-63 into the V slot (V is read for the last time)
      mbar_arrive_expect_tx(bar_g, G16 ? 16384 : 32768);
      tma_load_4d(sm + kB_V, &tm_g, bar_g, 0, h, t0, b);
      if (!G16) tma_load_4d(sm + kB_V + 8192, &tm_g, bar_g, 32, h, t0, b);
      ++g_issued;
      const uint32_t id = idesc_bf16(128, 64, false, true);
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtX1, sw128_desc(sZO + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024),
                 sw128_desc(sX0 + ks * 2048, 16384, 1024), id, ks > 0);
      mma_commit(bar_mma);
      bulk_wait_read_all();  // the staged dv is read before M and Po overwrite it
    }
    mma_wait();
    if (!ok) break;
    if (tid == 0) {
      // d 64-127 of the gate tile into the dZ halves (dZ is read for the last time)
      tma_load_4d(sm + kB_ZO, &tm_g, bar_g, 64, h, t0, b);
      if (!G16) tma_load_4d(sm + kB_ZO + 16384, &tm_g, bar_g, 96, h, t0, b);
    }
    {
      float x[16];
      tmem_ld16(tmem + lb + kBtX1 + cg * 16, x);
      if (row < 64) {
        // dA = -strict_lower(dZ U^T); dbeta part 2 = sum_j dA_rj (Kp Km^T)_rj; M = beta dA
        const int r = row;
        float kk[16];
        tmem_ld16(tmem + lb + kBtKQ + cg * 16, kk);
        const float br = bt[r];
        float s2 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float a = cg * 16 + i < r ? -x[i] : 0.f;
          s2 = fmaf(a, kk[i], s2);
          x[i] = br * a;
        }
        red[kR_DB2 + cg * 64 + r] = s2;
        store_chunks(sm + kB_T, r, cg * 2, x, 2);
      } else {
        // dP = lower(dO U^T): its diagonal kept apart, Po = the strictly lower part
        const int r = row - 64;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          if (j == r) dPd[r] = x[i];
          x[i] = j < r ? x[i] : 0.f;
        }
        store_chunks(sm + kB_P, r, cg * 2, x, 2);
      }
    }
    fence_async_shared();
    cta_sync();
    if (tid < 64) db2[tid] = red[kR_DB2 + tid] + red[kR_DB2 + 64 + tid] + red[kR_DB2 + 128 + tid] +
                             red[kR_DB2 + 192 + tid];
    if (tid >= 128 && tid < 256) {
      const int d = tid - 128;
      carry1[d] = red[kR_COL + d] + red[kR_COL + 128 + d] + red[kR_COL + 256 + d] + red[kR_COL + 384 + d];
    }
    // ---- the state-gradient update and the four dq / dk accumulators
    if (tid == 0) {
      const uint32_t idg = idesc_bf16(128, 128, true, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtG, sw128_desc(sZO + 8192 + ks * 2048, 16384, 1024),
                 sw128_desc(sKQ + 8192 + ks * 2048, 16384, 1024), idg, 1);
      const uint32_t idgn = idesc_bf16(128, 128, false, true, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtG, sw128_desc(sX1 + ks * 32, 16, 1024), sw128_desc(sKQ + ks * 2048, 16384, 1024),
                 idgn, 1);
      const uint32_t idq = idesc_bf16(128, 64, true, false);
      const uint32_t idmm = idesc_bf16(128, 64, true, true);
      const uint32_t idmmn = idesc_bf16(128, 64, true, true, true);
      // aQ^T = G~^T dO^T + Km^T Po^T
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtAQ, sw128_desc(sGI + ks * 2048, 16384, 1024),
                 sw128_desc(sZO + 8192 + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024), idq, ks > 0);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtAQ, sw128_desc(sKM + ks * 2048, 8192, 1024), sw128_desc(sP + ks * 32, 16, 1024), idq,
                 1);
      // aP^T = -G~^T dR^T + Km^T M^T
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtAP, sw128_desc(sGI + ks * 2048, 16384, 1024), sw128_desc(sX1 + ks * 2048, 16384, 1024),
                 idmmn, ks > 0);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtAP, sw128_desc(sKM + ks * 2048, 8192, 1024), sw128_desc(sT + ks * 32, 16, 1024), idq,
                 1);
      // aF^T = dG^^T U^T
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtAF, sw128_desc(sDG + ks * 2048, 16384, 1024), sw128_desc(sX0 + ks * 2048, 16384, 1024),
                 idmm, ks > 0);
      // aM^T = Qp^T Po + Kp^T M
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtAM, sw128_desc(sKQ + 8192 + ks * 2048, 16384, 1024),
                 sw128_desc(sP + ks * 2048, 16384, 1024), idmm, ks > 0);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtAM, sw128_desc(sKQ + ks * 2048, 16384, 1024), sw128_desc(sT + ks * 2048, 16384, 1024),
                 idmm, 1);
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // ---- E6
    if (tid == 0 && ci > 0) issue_main1(ci - 1);  // G~, T, dO have been read for the last time
    // the state gradient at the chunk's entry: dG diag(exp(lam)); into the
    // previous chunk's frame (diag(cf)) unless this is the first chunk
    if (ci > 0) {
      ok = __syncthreads_and(mbar_wait(bar_vec, vec_waited & 1));
      ++vec_waited;
      if (!ok) break;
    }
    {
      const float* el = vc + kVecElam;
      const float* cfp = vec(ci - 1) + kVecCf;
      float g[32];
      tmem_ld32(t_dg, g);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int d = cg * 32 + i;
        g[i] *= ci > 0 ? el[d] * cfp[d] : el[d];
      }
      tmem_st32(t_dg, g);
      if (ci > 0) write_dg(g);
    }
    ok = __syncthreads_and(mbar_wait(bar_g, g_waited & 1));
    ++g_waited;
    if (!ok) break;
    // gamma of this thread's elements: key dimension d = row, tokens r = 16 cg + i
    const int d = row;
    float gam[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)  // (a packed sequence's rows past its end hold the next one's gates)
      gam[i] = (!Packed || cg * 16 + i < n)
                   ? (G16 ? gate_elem16(sm, cg * 16 + i, d) : *gate_elem(sm, cg * 16 + i, d))
                   : 0.f;
#pragma unroll
    for (int i = 1; i < 16; ++i) gam[i] += gam[i - 1];
    red[kR_TOT + cg * 128 + d] = gam[15];
    __syncthreads();
    {
      float off = 0.f;
      for (int c2 = 0; c2 < cg; ++c2) off += red[kR_TOT + c2 * 128 + d];
      const float lm = vc[kVecLam + d];
#pragma unroll
      for (int i = 0; i < 16; ++i) gam[i] += off - lm;  // gamma - lam
    }
    float carry2 = 0.f, run = 0.f;
    const int hd = d >> 6, c16 = (d & 63) >> 3, e2 = (d & 7) * 2;
#pragma unroll
    for (int hh = 1; hh >= 0; --hh) {
      float ep[8], em[8], dgm[8], dk[8], a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        ep[i] = __expf(gam[8 * hh + i]);
        em[i] = __expf(-gam[8 * hh + i]);
      }
      float qp[8], kp[8], km[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = cg * 16 + 8 * hh + i, off = sw_row_off(r, c16) + e2;
        kp[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + kB_KQ + hd * 16384 + off));
        qp[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + kB_KQ + hd * 16384 + 8192 + off));
        km[i] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(sm + kB_KM + hd * 8192 + off));
      }
      tmem_ld8(tmem + lb + kBtAQ + cg * 16 + 8 * hh, a);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = cg * 16 + 8 * hh + i;
        const float dp = dPd[r];
        stage_bf16(sm + kB_X, r, d, fmaf(ep[i], a[i], dp * kp[i] * em[i]));  // dq
        dgm[i] = qp[i] * a[i];
        dk[i] = dp * qp[i] * em[i];
      }
      tmem_ld8(tmem + lb + kBtAP + cg * 16 + 8 * hh, a);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dk[i] = fmaf(ep[i], a[i], dk[i]);
        dgm[i] = fmaf(kp[i], a[i], dgm[i]);
      }
      tmem_ld8(tmem + lb + kBtAF + cg * 16 + 8 * hh, a);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        dk[i] = fmaf(em[i], a[i], dk[i]);
        dgm[i] = fmaf(-km[i], a[i], dgm[i]);
        carry2 = fmaf(km[i], a[i], carry2);
      }
      tmem_ld8(tmem + lb + kBtAM + cg * 16 + 8 * hh, a);
#pragma unroll
      for (int i = 7; i >= 0; --i) {
        const int r = cg * 16 + 8 * hh + i;
        dk[i] = fmaf(em[i], a[i], dk[i]);
        stage_bf16(sm + kB_X + 16384, r, d, dk[i]);  // dk
        run += fmaf(-km[i], a[i], dgm[i]);
        *gate_elem(sm, r, d) = run;  // suffix sum of dgamma within this thread's tokens
      }
    }
    red[kR_COL + cg * 128 + d] = run;
    red[kR_C2 + cg * 128 + d] = carry2;
    __syncthreads();
    if (tid == 0 && ci > 0) issue_main2(ci - 1);  // Kp|Qp and Km are read for the last time
    {
      float off = carry1[d];
      for (int c2 = 0; c2 < 4; ++c2) {
        off += red[kR_C2 + c2 * 128 + d];
        if (c2 > cg) off += red[kR_COL + c2 * 128 + d];
      }
      if (G16) {
        // dg straight to global memory in bf16 (32 lanes: 64 contiguous bytes per token)
        __nv_bfloat16* dg16 = reinterpret_cast<__nv_bfloat16*>(p.dg) +
                              (((size_t)b * p.T + t0) * p.H + h) * D + d;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (cg * 16 + i < n)
            dg16[(size_t)(cg * 16 + i) * p.H * D] = __float2bfloat16_rn(*gate_elem(sm, cg * 16 + i, d) + off);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) *gate_elem(sm, cg * 16 + i, d) += off;  // dg
      }
    }
    fence_async_shared();
    cta_sync();
    if (rowwise) {
      const size_t o0 = (((size_t)b * p.T + t0) * p.H + h) * D;
      store_rows_bf16(sm + kB_X, p.dq + o0, (size_t)p.H * D, n, tid, BT);
      store_rows_bf16(sm + kB_X + 16384, p.dk + o0, (size_t)p.H * D, n, tid, BT);
      if (!G16)
        for (int i = tid; i < n * 32; i += BT) {  // dg: 16-byte pieces of the fp32 rows
          const int r = i >> 5, c = i & 31;
          const float4 v = *reinterpret_cast<const float4*>(gate_elem(sm, r, c * 4));
          *reinterpret_cast<float4*>(p.dg + o0 + (size_t)r * p.H * D + c * 4) = v;
        }
    } else if (tid == 0) {
      tma_store_4d(&tm_dq, sm + kB_X, 0, h, t0, b);
      tma_store_4d(&tm_dq, sm + kB_X + 8192, 64, h, t0, b);
      tma_store_4d(&tm_dk, sm + kB_X + 16384, 0, h, t0, b);
      tma_store_4d(&tm_dk, sm + kB_X + 24576, 64, h, t0, b);
      if (!G16) {
        tma_store_4d(&tm_dg, sm + kB_V, 0, h, t0, b);
        tma_store_4d(&tm_dg, sm + kB_V + 8192, 32, h, t0, b);
        tma_store_4d(&tm_dg, sm + kB_ZO, 64, h, t0, b);
        tma_store_4d(&tm_dg, sm + kB_ZO + 16384, 96, h, t0, b);
      }
      bulk_commit_group();
    }
    if (tid < 64 && tid < n) p.dbeta[((size_t)b * p.T + t0 + tid) * p.H + h] = db1[tid] + db2[tid];
  }

  if (!ok) {
    if (tid == 0) {
      report_timeout();
      // let the loads still in flight land before the CTA exits (bounded)
      if (inflight >= 0) {
        if (parts < 2) issue_main2(inflight);
        mbar_wait(bar_load, load_phase, 10000);
      }
      for (int k = v_waited; k < v_issued; ++k) mbar_wait(bar_v, k & 1, 10000);
      for (int k = vec_waited; k < vec_issued; ++k) mbar_wait(bar_vec, k & 1, 10000);
      for (int k = g_waited; k < g_issued; ++k) mbar_wait(bar_g, k & 1, 10000);
    }
  } else if (p.dh0) {
    float g[32];
    tmem_ld32(t_dg, g);
#pragma unroll
    for (int i = 0; i < 32; ++i) p.dh0[((size_t)bh * D + cg * 32 + i) * D + row] = g[i];
  }
  if (tid == 0) bulk_wait_all();
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

// ---------------------------------------------------------------- host side

size_t skip_bytes(const Problem& p) { return align_up((size_t)num_seqs(p) * p.H * sizeof(int), 256); }
size_t ktiles_bytes(const Problem& p) { return align_up((size_t)max_chunks(p) * p.H * kKTBytes, 256); }
size_t kstates_bytes(const Problem& p) { return align_up((size_t)max_chunks(p) * p.H * 32768, 256); }

struct KdaLayout {
  int* skip;
  unsigned char* ktiles;
  __nv_bfloat16* states;  // saved context / backward only
  void* simt;             // the CUDA-core kernels' workspace (backward / saved context only)
};

KdaLayout layout(const Problem& p, bool with_bwd) {
  unsigned char* w = static_cast<unsigned char*>(p.ws);
  KdaLayout L{};
  L.skip = reinterpret_cast<int*>(w);
  L.ktiles = w + skip_bytes(p);
  if (with_bwd) {
    L.states = reinterpret_cast<__nv_bfloat16*>(L.ktiles + ktiles_bytes(p));
    L.simt = reinterpret_cast<unsigned char*>(L.states) + kstates_bytes(p);
  }
  return L;
}

// 4-D map over a [B, T, H, 128] fp32 tensor (the KDA gate and its gradient);
// box = 32 dimensions x 1 head x 64 tokens x 1 batch row, no swizzle (128-byte
// rows); rows past T read as zero and are not written.
// With a bf16 gate (g16) the box is 64 dimensions (the same 128-byte rows).
cudaError_t make_gate_map(CUtensorMap* m, const void* ptr, const Problem& p, int box_d = 0) {
  auto enc = get_encoder();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t es_bytes = p.g16 ? 2 : 4;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.H, (cuuint64_t)p.T, (cuuint64_t)p.B};
  cuuint64_t strides[3] = {(cuuint64_t)D * es_bytes, (cuuint64_t)p.H * D * es_bytes,
                           (cuuint64_t)p.T * p.H * D * es_bytes};
  cuuint32_t box[4] = {box_d ? (cuuint32_t)box_d : (p.g16 ? 64u : 32u), 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, p.g16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4,
                   const_cast<void*>(ptr), dims, strides, box, es,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_prep(const Problem& p, cudaStream_t s, const KdaLayout& L) {
  cudaError_t e = cudaMemsetAsync(L.skip, 0, (size_t)num_seqs(p) * p.H * sizeof(int), s);
  if (e != cudaSuccess) return e;
  CUtensorMap mk, mq, mg;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mq, p.q, p)) != cudaSuccess) return e;
  if ((e = make_gate_map(&mg, p.g, p, 128)) != cudaSuccess) return e;
  KdaPrepParams pp{p.g, p.beta, L.ktiles, L.skip, p.B, p.T, p.H, p.N, Seqs::of(p), p.nseq, p.g16};
  auto kern = p.cu_seqlens ? (p.g16 ? kda_tc_prep_kernel<true, true> : kda_tc_prep_kernel<true, false>)
                           : (p.g16 ? kda_tc_prep_kernel<false, true> : kda_tc_prep_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrepSmemBytes);
  if (e != cudaSuccess) return e;
  // an ordinary launch: it must follow the flags' reset in full
  prof_before(s);
  kern<<<(unsigned)(max_chunks(p) * p.H), PT, kPrepSmemBytes, s>>>(mk, mq, mg, pp);
  prof_after(s, kKdaPrep);
  return cudaGetLastError();
}

// Forward scan: the output (want_out) and/or the entry states.
cudaError_t launch_fwd(const Problem& p, cudaStream_t s, const KdaLayout& L, bool want_out,
                       __nv_bfloat16* states, int kernel_id) {
  CUtensorMap mv, mo;
  cudaError_t e;
  if ((e = make_token_map(&mv, p.v, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mo, want_out ? p.o : p.v, p)) != cudaSuccess) return e;
  KdaFwdParams fp{p.h0, want_out ? static_cast<__nv_bfloat16*>(p.o) : nullptr, want_out ? p.ht : nullptr,
                  states, L.ktiles, L.skip, p.B, p.T, p.H, p.N, Seqs::of(p)};
  auto kern = p.cu_seqlens ? kda_tc_fwd_kernel<true> : kda_tc_fwd_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kFwdSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  e = launch_overlapped(kern, (unsigned)(num_seqs(p) * p.H), FT, kFwdSmemBytes, s, mv, mo, fp);
  prof_after(s, kernel_id);
  return e;
}

}  // namespace

bool kda_tc_supported(const Problem& p) {
  return p.bf16 && p.kda && p.dk == D && p.dv == D && p.C == C;
}

// Forward workspace: the sequence flags and the per-chunk blocks.
size_t kda_tc_fwd_workspace(const Problem& p) { return skip_bytes(p) + ktiles_bytes(p); }

// Backward workspace and saved context: the forward's, the bf16 entry state of
// every chunk, and the CUDA-core kernels' workspace for flagged sequences.
size_t kda_tc_bwd_workspace(const Problem& p) {
  return skip_bytes(p) + ktiles_bytes(p) + kstates_bytes(p) + simt_bwd_workspace(p);
}

cudaError_t kda_tc_fwd(const Problem& p, cudaStream_t s, bool save) {
  const KdaLayout L = layout(p, save);
  cudaError_t e = launch_prep(p, s, L);
  if (e != cudaSuccess) return e;
  if ((e = launch_fwd(p, s, L, true, save ? L.states : nullptr, kKdaFwd)) != cudaSuccess) return e;
  // flagged sequences: the CUDA-core forward (saving its fp32 entry states)
  Problem q = p;
  q.ws = L.simt;
  return simt_fwd(q, s, save, L.skip);
}

// With saved, the workspace is a context filled by kda_tc_fwd(save) on the
// same inputs: the prep kernel and the states pass are not run again.
cudaError_t kda_tc_bwd(const Problem& p, cudaStream_t s, bool saved) {
  const KdaLayout L = layout(p, true);
  cudaError_t e;
  if (!saved) {
    if ((e = launch_prep(p, s, L)) != cudaSuccess) return e;
    if ((e = launch_fwd(p, s, L, false, L.states, kKdaStates)) != cudaSuccess) return e;
  }
  CUtensorMap mv, mdo, mg, mdq, mdk, mdv, mdg;
  if ((e = make_token_map(&mv, p.v, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdo, p.do_, p)) != cudaSuccess) return e;
  if ((e = make_gate_map(&mg, p.g, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdq, p.dq, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdk, p.dk_, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdv, p.dv_, p)) != cudaSuccess) return e;
  if ((e = make_gate_map(&mdg, p.dg, p)) != cudaSuccess) return e;
  KdaBwdParams bp{p.dht, L.ktiles, reinterpret_cast<const unsigned char*>(L.states), L.skip,
                  p.dbeta, p.dh0, static_cast<__nv_bfloat16*>(p.dq), static_cast<__nv_bfloat16*>(p.dk_),
                  static_cast<__nv_bfloat16*>(p.dv_), p.dg, p.B, p.T, p.H, p.N, Seqs::of(p)};
  auto kern = p.cu_seqlens ? (p.g16 ? kda_tc_bwd_kernel<true, true> : kda_tc_bwd_kernel<true, false>)
                           : (p.g16 ? kda_tc_bwd_kernel<false, true> : kda_tc_bwd_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  e = launch_overlapped(kern, (unsigned)(num_seqs(p) * p.H), BT, kBwdSmemBytes, s, mv, mdo, mg, mdq, mdk,
                        mdv, mdg, bp);
  prof_after(s, kKdaBwd);
  if (e != cudaSuccess) return e;
  // flagged sequences: the CUDA-core backward (with the entry states its
  // forward saved, or its own states pass)
  Problem q = p;
  q.ws = L.simt;
  return simt_bwd(q, s, saved, L.skip);
}

}  // namespace gdn
