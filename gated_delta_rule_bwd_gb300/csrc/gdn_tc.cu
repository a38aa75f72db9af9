// Tensor-core (tcgen05 / TMEM / TMA) kernels for the GDN mixer: bf16 inputs,
// dk = dv = 128, chunk C = 64, fp32 state and accumulation.
//
// Notation (gamma = within-chunk cumulative log gate, e = exp(gamma),
// f = exp(gamma_last - gamma), eC = exp(gamma_last), Gam[r][j] =
// exp(gamma_r - gamma_j)):
//   A = strict_lower(beta_r K K^T o Gam),  T = (I + A)^-1,
//   P = lower(Q K^T o Gam),  W = T diag(beta e) K,  U = T diag(beta)(V - eK H).
//
// Three kernels:
//   solve     one CTA per chunk, all chunks at once: MMA1 K K^T, A, and the
//             blocked triangular solve; writes T as a bf16 64 x 64 tile in
//             MMA-operand layout (8 KB per chunk) to the workspace.
//   forward   one CTA per (batch, head) walking its chunks in order.  The
//             state is held transposed, G = H^T (dv x dk), fp32 in TMEM with
//             a bf16 copy in shared memory as the MMA operand.  Per chunk:
//               MMA   Q K^T -> P
//               MMA2  W^T = K^T T'^T, T' = T diag(beta e)
//               MMA3  U^T = V^T T''^T - G W^T, T'' = T diag(beta)
//               MMA4  O = (eQ) G^T + P U          (M = 64: rows are tokens)
//               MMA5  G <- eC G + (U diag(f))^T K
//             The output rows and, when asked, every chunk's bf16 entry state
//             (for the backward pass: in states mode, which skips P and O, or
//             alongside the output for a saved context) leave the CTA by
//             TMA / bulk copies of their shared-memory tiles.
//   backward  the reverse chunk scan (described at its kernel).
//
// The TMA tiles of K and V serve both as K-major operands (rows = tokens) and,
// through MN-major descriptors, as their own transposes, so nothing is
// transposed in software.  MMAs are issued by one thread and complete on an
// mbarrier; every wait is bounded and a timeout is reported through the device
// status word instead of hanging.

#include <algorithm>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn.h"
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"
#include "tc_common.cuh"

namespace gdn {

// The status words of the bounded device-side waits: this file's and the KDA
// kernels'; a timeout recorded in either is reported.
cudaError_t read_and_clear_device_status(int* status) {
  int a = GDN_OK, b = GDN_OK, c = GDN_OK;
  cudaError_t e = tc::read_and_clear_file_status(&a);
  if (e == cudaSuccess) e = kda_read_and_clear_status(&b);
  if (e == cudaSuccess) e = nb_read_and_clear_status(&c);
  if (e != cudaSuccess) return e;
  *status = a != GDN_OK ? a : (b != GDN_OK ? b : c);
  return cudaSuccess;
}

namespace {

using namespace tc;

// ---------------------------------------------------------------- forward shared memory
// Offsets in bytes from a 1024-aligned base.  Two K|Q stages hold
// [K d0-63 | Q d0-63 | K d64-127 | Q d64-127] (8 KB each) so that [K;Q] is one
// 128-row operand, each with the chunk's T tile; V is single-buffered (only
// the preparation reads it).
constexpr int kF_KQ = 0;                   // 2 x 32 KB
constexpr int kF_V = 65536;                // 16 KB
constexpr int kF_G = 81920;                // G bf16, K-major [c][d], 2 x 16 KB
constexpr int kF_W = 114688;               // W, MN-major rows d, 64 r   (16 KB)
constexpr int kF_P = 131072;               // 2 x P [r][j]                (8 KB each)
constexpr int kF_T1 = 147456;              // T' = T diag(beta e) [r][j]  (8 KB)
constexpr int kF_T0 = 155648;              // T'' = T diag(beta) [r][j]   (8 KB)
constexpr int kF_U = 163840;               // U^T [c][j] K-major          (16 KB)
constexpr int kF_TR = 180224;              // 2 x T [r][j] as written by the solve kernel (8 KB each)
constexpr int kF_GATE = kF_TR + 2 * 8192;
constexpr int kGateBlock = 1600;           // gamma, e, f, beta, er, ie [64] each, eC, fast; two blocks
constexpr int kF_GRAW = kF_GATE + 2 * kGateBlock;  // 2 x 128 raw g, beta (prefetch)
constexpr int kF_BAR = kF_GRAW + 2 * 512;
constexpr int kSmemBytes = kF_BAR + 128 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// TMEM columns of the forward kernel: K K^T | Q K^T, W^T, two U^T buffers,
// O (M = 64 rows: token r in lane 32 (r / 16) + r % 16, 128 columns) and the
// fp32 state G (128 columns).
constexpr uint32_t kTmKQ = 0, kTmW = 64, kTmU0 = 128, kTmO = 256, kTmG = 384, kTmCols = 512;

struct FwdParams {
  const float* g;
  const float* beta;
  const float* h0;
  __nv_bfloat16* o;
  float* ht;
  __nv_bfloat16* states;  // optional: bf16 G tile of every chunk's entry state
                          // ([B*H][N][32 KB], shared-memory layout)
  const unsigned char* tiles;  // T of every chunk ([B*H][N][8 KB], from the solve kernel)
  int B, T, H, N;
  Seqs sq;  // the call's sequences (a batch, or packed sequences)
  // Segments (long sequences): with seg_chunks > 0 each CTA runs seg_chunks
  // chunks of one sequence (CTA = sequence * nseg + segment); h0 and ht are
  // then per segment ([B*H*nseg][dk][dv]).
  int seg_chunks;
  int v_zero;       // treat V as zero (the segment's transition map)
  int h0_identity;  // start from H = I instead of h0 (dk = dv)
};

// ---------------------------------------------------------------- forward kernel
//
// Warp-specialised, 512 threads.  Warps 8-15 (the preparation group) run the
// state-independent part of chunk c+1: the gates, T' and T'' from the loaded
// T tile, Q K^T and P, MMA2/MMA3a.  Warps 0-7 (the chain group) meanwhile run chunk c:
// the W tile from W^T, the row scalings eQ and fK, MMA3b/MMA4a, U^T,
// MMA4b/MMA5, the output and the next state tile.
// Warp w reads TMEM lane quadrant w % 4 and handles column half (w / 4) % 2
// of every tile.  Hand-offs use mbarriers; each group synchronises internally
// with its own named barrier.  The fp32 state lives in TMEM: before MMA5 the
// chain scales it by eC and MMA5 accumulates (U diag f)^T K onto it.

constexpr int FT = 512;
// Gates of one chunk, computed by one warp from the lane's two log gates
// (rows lane and lane + 32) and betas: gamma = inclusive cumsum of g,
// e = exp(gamma), f = exp(gamma_last - gamma), eC = exp(gamma_last).  For the
// decay factors Gam[r][j] = exp(gamma_r - gamma_j) it also writes
// er = exp(gamma - gref) and ie = exp(gref - gamma) with gref the middle of
// the chunk's gamma range; when that range is below 80 the product er_r ie_j
// equals Gam[r][j] without overflow and *fast is set, otherwise the exact
// per-element exponential is used.
struct GateView {
  float *gam, *ee, *ff, *bt, *er, *ie, *eC, *fast;
};

__device__ __forceinline__ void chunk_gates(const GateView& G, float g0, float g1, float b0,
                                            float b1, int lane) {
  G.bt[lane] = b0;
  G.bt[lane + 32] = b1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float a0 = __shfl_up_sync(0xffffffffu, g0, off);
    const float a1 = __shfl_up_sync(0xffffffffu, g1, off);
    if (lane >= off) g0 += a0, g1 += a1;
  }
  g1 += __shfl_sync(0xffffffffu, g0, 31);
  const float gl = __shfl_sync(0xffffffffu, g1, 31);
  float mx = fmaxf(g0, g1), mn = fminf(g0, g1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
  }
  const float gref = 0.5f * (mx + mn);
  G.gam[lane] = g0;
  G.gam[lane + 32] = g1;
  G.ee[lane] = __expf(g0);
  G.ee[lane + 32] = __expf(g1);
  G.ff[lane] = __expf(gl - g0);
  G.ff[lane + 32] = __expf(gl - g1);
  G.er[lane] = __expf(g0 - gref);
  G.er[lane + 32] = __expf(g1 - gref);
  G.ie[lane] = __expf(gref - g0);
  G.ie[lane + 32] = __expf(gref - g1);
  if (lane == 0) {
    *G.eC = __expf(gl);
    *G.fast = (mx - mn < 80.f) ? 1.f : 0.f;
  }
}

// The gates of the next chunk are prefetched by one warp with asynchronous
// 4-byte copies into a raw block [g rows 0-31 | g rows 32-63 | beta rows 0-31 |
// beta rows 32-63] (128 floats; rows past the sequence end read as zero), so
// that their global-memory latency stays off the chunk's critical path.
__device__ __forceinline__ void prefetch_gates(float* raw, const float* g, const float* beta,
                                               size_t row0, int n, int H, int h, int lane) {
  const size_t base = row0 * H + h;
  const size_t o0 = lane < n ? base + (size_t)lane * H : base;
  const size_t o1 = lane + 32 < n ? base + (size_t)(lane + 32) * H : base;
  cp_async4(raw + lane, g + o0, lane < n);
  cp_async4(raw + 32 + lane, g + o1, lane + 32 < n);
  cp_async4(raw + 64 + lane, beta + o0, lane < n);
  cp_async4(raw + 96 + lane, beta + o1, lane + 32 < n);
  cp_async_commit();
}

// chunk_gates from a prefetched raw block (each lane reads only what it copied)
__device__ __forceinline__ void chunk_gates_raw(const GateView& G, const float* raw, int lane) {
  cp_async_wait_all();
  chunk_gates(G, raw[lane], raw[32 + lane], raw[64 + lane], raw[96 + lane], lane);
}

// Decayed row: v[i] <- v[i] * Gam[r][j0 + i] for j0 + i <= r (or < r when
// strict), 0 above; n columns.
template <int n>
__device__ __forceinline__ void decay_row(float (&v)[n], const GateView& G, int r, int j0,
                                          bool strict, float scale) {
  if (*G.fast != 0.f) {
    const float a = G.er[r] * scale;
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const int j = j0 + i;
      v[i] = (strict ? j < r : j <= r) ? v[i] * a * G.ie[j] : 0.f;
    }
  } else {
    const float gr = G.gam[r];
#pragma unroll
    for (int i = 0; i < n; ++i) {
      const int j = j0 + i;
      v[i] = (strict ? j < r : j <= r) ? scale * v[i] * __expf(gr - G.gam[j]) : 0.f;
    }
  }
}

template <bool NoDelta, bool Packed>
__global__ void __launch_bounds__(FT, 1)
gdn_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, half = (warp >> 2) & 1, grp = warp >> 3;
  const int row = quad * 32 + lane;    // TMEM lane / tile row owned by this thread
  // this CTA's sequence and chunks [c0, c0 + NL) (the whole sequence unless
  // segmented; segments are used for batches only)
  const int nseg = p.seg_chunks ? (p.N + p.seg_chunks - 1) / p.seg_chunks : 1;
  const int seg = blockIdx.x % nseg, bh = blockIdx.x / nseg, sq_s = bh / p.H, h = bh % p.H;
  const int c0 = seg * p.seg_chunks;
  int b = 0, tb = 0, slen = 0, NL = 0;  // batch row, first token, length, chunks (after the wait)
  const size_t st_idx = (size_t)bh * nseg + seg;  // index of h0 / ht
  const bool has_v = !p.v_zero;

  uint64_t* bar_kq = reinterpret_cast<uint64_t*>(sm + kF_BAR);  // [2] K|Q stage loaded
  uint64_t* bar_v = bar_kq + 2;                                  // V loaded
  uint64_t* bar_p = bar_kq + 3;                                  // preparation MMAs done
  uint64_t* bar_s = bar_kq + 4;                                  // chain MMAs done
  uint64_t* bar_pd = bar_kq + 5;                                 // preparation of a chunk done
  uint64_t* bar_wf = bar_kq + 6;                                 // W^T TMEM read by the chain
  uint64_t* bar_p1 = bar_kq + 7;                                 // preparation MMA1 done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_kq + 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* cnt = reinterpret_cast<int*>(tmem_slot + 2);  // [0..1] kq issued, [2..3] kq waited, [4] v issued, [5] v waited, [6] early MMA1

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(&bar_kq[i], 1);
    *abort_flag = 0;
    for (int i = 0; i < 7; ++i) cnt[i] = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
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
  grid_dep_wait();  // the previous kernel's results (and its reads of what this one writes)
  grid_dep_launch();
  {
    int nch;
    p.sq.get_t<Packed>(sq_s, b, tb, slen, nch);
    NL = p.seg_chunks ? min(p.seg_chunks, nch - c0) : nch;
  }

  auto load_kq = [&](int ci) {
    const int st = ci & 1;
    unsigned char* dst = sm + kF_KQ + st * 32768;
    mbar_arrive_expect_tx(&bar_kq[st], 32768 + (NoDelta ? 0 : 8192));
    const int t0 = tb + (c0 + ci) * C;
    tma_load_4d(dst + 0, &tm_k, &bar_kq[st], 0, h, t0, b);
    tma_load_4d(dst + 8192, &tm_q, &bar_kq[st], 0, h, t0, b);
    tma_load_4d(dst + 16384, &tm_k, &bar_kq[st], 64, h, t0, b);
    tma_load_4d(dst + 24576, &tm_q, &bar_kq[st], 64, h, t0, b);
    if (!NoDelta)
      bulk_load(sm + kF_TR + st * 8192, p.tiles + rec_bh<Packed>(p.sq, p.N, bh, sq_s, h, c0 + ci) * 8192, 8192, &bar_kq[st]);
    cnt[st] += 1;
  };
  auto load_v = [&](int ci) {
    mbar_arrive_expect_tx(bar_v, 16384);
    const int t0 = tb + (c0 + ci) * C;
    tma_load_4d(sm + kF_V, &tm_v, bar_v, 0, h, t0, b);
    tma_load_4d(sm + kF_V + 8192, &tm_v, bar_v, 64, h, t0, b);
    cnt[4] += 1;
  };
  auto state_dst = [&](int ci) -> unsigned char* {
    return p.states ? reinterpret_cast<unsigned char*>(p.states) + rec_bh<Packed>(p.sq, p.N, bh, sq_s, h, c0 + ci) * (size_t)32768
                    : nullptr;
  };
  const bool want_o = p.o != nullptr;

  if (tid == 0 && NL > 0) {
    load_kq(0);
    if (NL > 1) load_kq(1);
    if (has_v) load_v(0);
  }
  bool ok = true;

  if (grp == 0) {
    // ============================== chain group ==============================
    const int gt = tid;
    // initial state: fp32 in TMEM and the bf16 tile; this thread: d in [64 half, 64 half + 64)
    {
      float v[32];
#pragma unroll
      for (int q32 = 0; q32 < 2; ++q32) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int d = half * 64 + q32 * 32 + i;
          v[i] = p.h0_identity ? (d == row ? 1.f : 0.f)
                               : (p.h0 ? p.h0[(st_idx * D + d) * D + row] : 0.f);
        }
        tmem_st32(tmem + lane_base + kTmG + half * 64 + q32 * 32, v);
        store_chunks(sm + kF_G + half * 16384, row, q32 * 4, v, 4);
      }
    }
    fence_async_shared();
    group_sync_tc(kBarChain);
    if (gt == 0 && p.states && NL > 0) {
      // states mode: the tile is also chunk 0's entry state in the workspace
      bulk_store(state_dst(0), sm + kF_G, 32768);
      bulk_commit_group();
    }
    uint32_t s_phase = 0;
    for (int ci = 0; ci < NL; ++ci) {
      const int s = ci & 1, t0 = tb + (c0 + ci) * C, nrow = min(C, slen - (c0 + ci) * C);
      const float* gates = reinterpret_cast<const float*>(sm + kF_GATE + s * kGateBlock);  // eC at [384]
      ok = group_and(kBarChain, kGroup, mbar_wait(bar_pd, ci & 1) && !*abort_flag);
      if (!ok) break;
      tc_fence_after();
      if (!NoDelta) {
        // W^T (TMEM) -> W tile, MN-major: row d holds W[0..63][d]
        float w[32];
        tmem_ld32(tmem + lane_base + kTmW + half * 32, w);
        store_chunks(sm + kF_W, row, half * 4, w, 4);
      }
      {
        // rows of this chunk's stage: Q by e (for MMA4a), K by f (for MMA5);
        // the preparation's MMA1 and MMA2 are done with both
        unsigned char* stc = sm + kF_KQ + s * 32768;
        const float* ge = gates + 64;
        const float* gf = gates + 128;
        if (want_o) {
          scale_rows(stc + 8192, 64, ge, gt, kGroup);
          scale_rows(stc + 24576, 64, ge, gt, kGroup);
        }
        scale_rows(stc, 64, gf, gt, kGroup);
        scale_rows(stc + 16384, 64, gf, gt, kGroup);
      }
      if (ci == 0) {
        // G <- eC G  (MMA5 accumulates onto it; for later chunks the previous
        // chunk's last epilogue does this)
        const float ec = gates[384];
        float v[32];
#pragma unroll
        for (int q32 = 0; q32 < 2; ++q32) {
          const uint32_t ta = tmem + lane_base + kTmG + half * 64 + q32 * 32;
          tmem_ld32(ta, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= ec;
          tmem_st32(ta, v);
        }
      }
      fence_async_shared();
      group_sync_tc(kBarChain);
      if (gt == 0) mbar_arrive(bar_wf);  // W^T has been copied: the next MMA2 may run
      const uint32_t st_off = kF_KQ + s * 32768;  // this chunk's K|Q stage
      const uint32_t tmU = kTmU0 + 64 * s;
      if (gt == 0) {
        // MMA3b: U^T += -G W^T (A: G K-major M=c K=d; B: W MN-major N=r K=d);
        // without the delta rule U = diag(beta) V holds no state term
        const uint32_t id3 = idesc_bf16(128, 64, false, true, true);
        if (!NoDelta) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16(tmem + tmU, desc_at(dK0, kF_G + (ks / 4) * 16384 + (ks % 4) * 32),
                     desc_at(dM0, kF_W + ks * 2048), id3, has_v || ks > 0);
        }
        // MMA4a: O = (eQ) G^T  (M=64: A = eQ rows r, K=d; B = G tile rows c, K=d)
        const uint32_t id4 = idesc_bf16(64, 128, false, false);
        if (want_o) {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
            mma_bf16(tmem + kTmO, desc_at(dK0, st_off + 8192 + off), desc_at(dK0, kF_G + off), id4, ks > 0);
          }
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
        // MMA4b: O += P U  (A = P rows r, K=j; B = U^T tile rows c, K=j)
        const uint32_t id4 = idesc_bf16(64, 128, false, false);
        if (want_o) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + kTmO, desc_at(dK0, kF_P + s * 8192 + ks * 32), desc_at(dK0, kF_U + ks * 32), id4, 1);
        }
        // MMA5: G += U^T (f K)  (B: K tile, rows scaled by f, MN-major N=d, K=j)
        const uint32_t id5 = idesc_bf16(128, 128, false, true);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tmem + kTmG, desc_at(dK0, kF_U + ks * 32), desc_at(dM0, st_off + ks * 2048), id5, 1);
        mma_commit(bar_s);
        bulk_wait_read_all();  // the last entry-state copy has read the tile E5 rewrites next
      }
      ok = group_and(kBarChain, kGroup, mbar_wait(bar_s, s_phase));
      s_phase ^= 1;
      tc_fence_after();
      if (!ok) break;
      if (gt == 0 && ci + 2 < NL) load_kq(ci + 2);  // this stage is no longer read
      if (want_o) {
        // O row r = 16 quad + lane (lanes 0-15 of each quadrant), columns 64 half + [0, 64),
        // staged in the U^T tile's slot (its products are done) for a TMA store
        const int r = quad * 16 + lane;
#pragma unroll
        for (int q32 = 0; q32 < 2; ++q32) {
          float v[32];
          tmem_ld32(tmem + lane_base + kTmO + half * 64 + q32 * 32, v);
          if (lane < 16) store_chunks(sm + kF_U + half * 8192, r, q32 * 4, v, 4);
        }
      }
      {
        // bf16 copy of the next chunk's entry state; then G <- eC G with the
        // next chunk's eC (its gates are ready: they precede its hand-over)
        const bool more = ci + 1 < NL;
        unsigned char* dst = more ? state_dst(ci + 1) : nullptr;
        const float ecn =
            more ? reinterpret_cast<const float*>(sm + kF_GATE + ((ci + 1) & 1) * kGateBlock)[384] : 1.f;
        float v[32];
#pragma unroll
        for (int q32 = 0; q32 < 2; ++q32) {
          const uint32_t ta = tmem + lane_base + kTmG + half * 64 + q32 * 32;
          tmem_ld32(ta, v);
          store_chunks(sm + kF_G + half * 16384, row, q32 * 4, v, 4);
          if (more) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= ecn;
            tmem_st32(ta, v);
          }
        }
        fence_async_shared();
        group_sync_tc(kBarChain);
        // the output rows: a tensor store (rows past T are not written), or row
        // by row for a packed sequence's partial last chunk
        const bool rowwise = Packed && want_o && nrow < C;
        if (rowwise)
          store_rows_bf16(sm + kF_U, p.o + (((size_t)b * p.T + t0) * p.H + h) * D, (size_t)p.H * D, nrow,
                          gt, kGroup);
        if (gt == 0 && (dst || want_o)) {
          if (dst) bulk_store(dst, sm + kF_G, 32768);  // the next chunk's entry state to the workspace
          if (want_o && !rowwise) {
            tma_store_4d(&tm_o, sm + kF_U, 0, h, t0, b);
            tma_store_4d(&tm_o, sm + kF_U + 8192, 64, h, t0, b);
          }
          bulk_commit_group();
        }
      }
    }
    if (gt == 0) bulk_wait_all();  // entry-state copies complete (and their tile reads)
    if (!ok) *abort_flag = 1;
    if (ok && p.ht) {
      float v[32];
#pragma unroll
      for (int q32 = 0; q32 < 2; ++q32) {
        tmem_ld32(tmem + lane_base + kTmG + half * 64 + q32 * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          p.ht[(st_idx * D + half * 64 + q32 * 32 + i) * D + row] = v[i];
      }
    }
  } else {
    // =========================== preparation group ===========================
    const int pt = tid - kGroup;
    auto psync = [&]() { group_sync(kBarPrep, kGroup); };
    float* graw = reinterpret_cast<float*>(sm + kF_GRAW);
    auto load_gates = [&](int ci) {
      const int t = (c0 + ci) * C;
      prefetch_gates(graw + (ci & 1) * 128, p.g, p.beta, (size_t)b * p.T + tb + t, min(C, slen - t), p.H,
                     h, lane);
    };
    // Warp 9 (which issues nothing) computes each chunk's gates one chunk
    // ahead, at the end of the previous chunk's preparation, from raw values
    // prefetched one more chunk ahead; chunk 0's here.
    auto gate_view = [&](int ci) {
      float* gb = reinterpret_cast<float*>(sm + kF_GATE + (ci & 1) * kGateBlock);
      return GateView{gb, gb + 64, gb + 128, gb + 192, gb + 256, gb + 320, gb + 384, gb + 385};
    };
    if (warp == 9 && NL > 0) {
      load_gates(0);
      chunk_gates_raw(gate_view(0), graw, lane);
      if (NL > 1) load_gates(1);
    }
    volatile int* early_mma1 = cnt + 6;
    if (pt == 0) *early_mma1 = 0;
    auto issue_mma1 = [&](int cn) {
      // MMA1: [K;Q] K^T, M=128 N=64 K=128 on the stage of chunk cn
      const uint32_t kq = kF_KQ + (cn & 1) * 32768;
      const uint32_t idesc = idesc_bf16(128, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        mma_bf16(tmem + kTmKQ, desc_at(dK0, kq + off), desc_at(dK0, kq + off), idesc, ks > 0);
      }
      mma_commit(bar_p1);
    };
    uint32_t p_phase = 0;
    for (int ci = 0; ci < NL; ++ci) {
      const int s = ci & 1;
      float* gates = reinterpret_cast<float*>(sm + kF_GATE + s * kGateBlock);
      const GateView GV{gates, gates + 64, gates + 128, gates + 192, gates + 256, gates + 320,
                        gates + 384, gates + 385};
      float* ee = GV.ee;
      float* bt = GV.bt;
      ok = group_and(kBarPrep, kGroup, mbar_wait(&bar_kq[s], (ci >> 1) & 1) && !*abort_flag);
      if (!ok) break;
      if (pt == 0) cnt[2 + s] += 1;
      if (want_o && pt == 0 && !*early_mma1) issue_mma1(ci);
      {
        // T' = T diag(beta e) and T'' = T diag(beta): columns of the loaded T
        // tile (same swizzled layout in and out).  This thread: 16-byte column
        // chunk c8 of rows r and r + 32.
        const int c8 = pt & 7, r0 = pt >> 3;
        float sb[8], sbe[8];
        {
          const float4 b0 = *reinterpret_cast<const float4*>(bt + c8 * 8);
          const float4 b1 = *reinterpret_cast<const float4*>(bt + c8 * 8 + 4);
          const float4 e0 = *reinterpret_cast<const float4*>(ee + c8 * 8);
          const float4 e1 = *reinterpret_cast<const float4*>(ee + c8 * 8 + 4);
          const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
          const float e8[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            sb[k] = bb[k];
            sbe[k] = bb[k] * e8[k];
          }
        }
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const int off = sw_row_off(r0 + 32 * rr, c8);
          uint4 raw = make_uint4(0u, 0u, 0u, 0u);
          if (NoDelta) {
            // T = I: the row's diagonal element, if it falls in this column chunk
            const int rw = r0 + 32 * rr;
            if ((rw >> 3) == c8) {
              __nv_bfloat16* e = reinterpret_cast<__nv_bfloat16*>(&raw);
              e[rw & 7] = __float2bfloat16_rn(1.f);
            }
          } else {
            raw = *reinterpret_cast<const uint4*>(sm + kF_TR + s * 8192 + off);
          }
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
          uint4 o1, o0;
          uint32_t* w1 = reinterpret_cast<uint32_t*>(&o1);
          uint32_t* w0 = reinterpret_cast<uint32_t*>(&o0);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 t = __bfloat1622float2(h2[k]);
            __nv_bfloat162 x0 = __floats2bfloat162_rn(t.x * sb[2 * k], t.y * sb[2 * k + 1]);
            __nv_bfloat162 x1 = __floats2bfloat162_rn(t.x * sbe[2 * k], t.y * sbe[2 * k + 1]);
            w0[k] = *reinterpret_cast<uint32_t*>(&x0);
            w1[k] = *reinterpret_cast<uint32_t*>(&x1);
          }
          *reinterpret_cast<uint4*>(sm + kF_T1 + off) = o1;
          *reinterpret_cast<uint4*>(sm + kF_T0 + off) = o0;
        }
      }
      if (want_o) {
        ok = group_and(kBarPrep, kGroup, mbar_wait(bar_p1, ci & 1));
        tc_fence_after();
        if (!ok) break;
        // P (TMEM lanes 64-127): 32 columns per thread; quadrant 2 holds rows
        // 0-31, whose columns 32-63 are zero
        if (row >= 64) {
          const int r = row - 64;
          float v[32];
          if (quad == 2 && half == 1) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          } else {
            tmem_ld32(tmem + lane_base + kTmKQ + half * 32, v);
            decay_row(v, GV, r, half * 32, false, 1.f);
          }
          store_chunks(sm + kF_P + s * 8192, r, half * 4, v, 4);
        }
      }
      if (has_v) {
        ok = group_and(kBarPrep, kGroup, mbar_wait(bar_v, ci & 1));
        if (!ok) break;
        if (pt == 0) cnt[5] += 1;
      }
      if (ci > 0) {
        // the chain has copied the previous chunk's W^T out of TMEM
        ok = group_and(kBarPrep, kGroup, mbar_wait(bar_wf, (ci - 1) & 1));
        if (!ok) break;
      }
      fence_async_shared();
      tc_fence_before();
      psync();
      tc_fence_after();
      if (pt == 0) {
        // MMA2: W^T = K^T T'^T  (A: K tile MN-major, M=d; B: T' K-major, N=r)
        const uint32_t id2 = idesc_bf16(128, 64, true, false);
        const uint32_t st_off = kF_KQ + s * 32768;
        if (!NoDelta) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + kTmW, desc_at(dM0, st_off + ks * 2048), desc_at(dK0, kF_T1 + ks * 32), id2, ks > 0);
        }
        // MMA3a: U^T = V^T T''^T  (A: V tile MN-major, M=c; B: T'' K-major, N=r)
        if (has_v) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tmem + kTmU0 + 64 * s, desc_at(dV0, kF_V + ks * 2048), desc_at(dK0, kF_T0 + ks * 32), id2,
                     ks > 0);
        }
        mma_commit(bar_p);
      }
      if (warp == 9 && ci + 1 < NL) {
        // gates of the next chunk: its block was last read by the chain for
        // chunk ci - 1, which has released it (the w_free wait above)
        chunk_gates_raw(gate_view(ci + 1), graw + ((ci + 1) & 1) * 128, lane);
        if (ci + 2 < NL) load_gates(ci + 2);
      }
      ok = group_and(kBarPrep, kGroup, mbar_wait(bar_p, p_phase));
      p_phase ^= 1;
      tc_fence_after();
      if (!ok) break;
      if (has_v && pt == 0 && ci + 1 < NL) load_v(ci + 1);
      if (want_o && pt == 0) {
        // the Q K^T columns are free again: start the next chunk's MMA1 now if
        // its tiles have landed (otherwise it is issued at the top of that chunk)
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
      // let tile loads still in flight land before the CTA exits (bounded)
      for (int st = 0; st < 2; ++st)
        for (int k = cnt[2 + st]; k < cnt[st]; ++k) mbar_wait(&bar_kq[st], k & 1, 10000);
      for (int k = cnt[5]; k < cnt[4]; ++k) mbar_wait(bar_v, k & 1, 10000);
    }
  }
  cp_async_wait_all();  // no gate prefetch may still be writing shared memory at exit
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

// ---------------------------------------------------------------- solve kernel
//
// One CTA of 256 threads per chunk, every chunk of every sequence at once (the
// solve does not depend on the state):
//   MMA1  K K^T (M = 64: row r in TMEM lane 32 (r / 16) + r % 16)
//         A = strict_lower(beta_r K K^T o Gam)            (fp32, shared memory)
//         T = (I + A)^-1                                   (solve_unit_lower)
// T is written as a bf16 64 x 64 tile, zero above the diagonal, in the
// K-major 128-byte-swizzled layout of an MMA operand, so that the scans copy
// it into shared memory unchanged (8 KB per chunk, [B*H][N] order).
// About 53 KB of shared memory and 64 TMEM columns: four CTAs per SM.

constexpr int ST = 256;
constexpr int kS_K = 0;                            // [K d0-63 | K d64-127]; solve scratch after MMA1
constexpr int kS_A = 16384;                        // A fp32 [64][kLdF]
constexpr int kS_T = kS_A + 64 * kLdF * 4;         // T fp32 [64][kLdF]
constexpr int kS_GATE = kS_T + 64 * kLdF * 4;      // one gate block
constexpr int kS_BAR = kS_GATE + kGateBlock;
constexpr int kSolveSmemBytes = kS_BAR + 64 + 1024;  // + alignment slack
static_assert(kSolveScratch * 4 <= 16384, "solve scratch fits the K tile");
static_assert(4 * (kSolveSmemBytes + 1024) <= 228 * 1024, "four solve CTAs per SM");

struct SolveParams {
  const float* g;
  const float* beta;
  unsigned char* tiles;  // 8 KB per chunk record
  int B, T, H, N;
  Seqs sq;
  int nseq;
};

template <bool Packed>
__global__ void __launch_bounds__(ST)
gdn_tc_solve_kernel(const __grid_constant__ CUtensorMap tm_k, SolveParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, half = warp >> 2;
  float* gates = reinterpret_cast<float*>(sm + kS_GATE);
  const GateView GV{gates, gates + 64, gates + 128, gates + 192, gates + 256, gates + 320,
                    gates + 384, gates + 385};
  float* Am = reinterpret_cast<float*>(sm + kS_A);
  float* Tm = reinterpret_cast<float*>(sm + kS_T);
  float* Sm = reinterpret_cast<float*>(sm + kS_K);
  uint64_t* bar_ld = reinterpret_cast<uint64_t*>(sm + kS_BAR);
  uint64_t* bar_mma = bar_ld + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);

  grid_dep_wait();  // the previous kernel's results (and its reads of what this one writes)
  grid_dep_launch();
  int sqi, h, ci, b, tb, len, nch;
  if (!p.sq.chunk_of(blockIdx.x, p.nseq, sqi, h, ci)) return;  // past the last packed chunk
  p.sq.get_t<Packed>(sqi, b, tb, len, nch);
  const int t0 = tb + ci * C, n = min(C, len - ci * C);
  if (tid == 0) {
    mbar_init(bar_ld, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar_ld, 16384);
    tma_load_4d(sm + kS_K, &tm_k, bar_ld, 0, h, t0, b);
    tma_load_4d(sm + kS_K + 8192, &tm_k, bar_ld, 64, h, t0, b);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 64);
    tmem_relinquish();
  }
  if (warp == 1) {
    const size_t base = ((size_t)b * p.T + t0) * p.H + h;
    const float g0 = lane < n ? p.g[base + (size_t)lane * p.H] : 0.f;
    const float g1 = lane + 32 < n ? p.g[base + (size_t)(lane + 32) * p.H] : 0.f;
    const float b0 = lane < n ? p.beta[base + (size_t)lane * p.H] : 0.f;
    const float b1 = lane + 32 < n ? p.beta[base + (size_t)(lane + 32) * p.H] : 0.f;
    chunk_gates(GV, g0, g1, b0, b1, lane);
  }
  cta_sync();
  const uint32_t tmem = *tmem_slot;
  bool loaded = __syncthreads_and(mbar_wait(bar_ld, 0));
  bool ok = loaded;
  if (ok) {
    if (tid == 0) {
      tc_fence_after();
      const uint64_t dk = sw128_desc(smem_u32(sm + kS_K), 16, 1024);
      const uint32_t id = idesc_bf16(64, 64, false, false);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 8192 + (ks % 4) * 32;
        mma_bf16(tmem, desc_at(dk, off), desc_at(dk, off), id, ks > 0);
      }
      mma_commit(bar_mma);
    }
    ok = __syncthreads_and(mbar_wait(bar_mma, 0));
    tc_fence_after();
  }
  if (ok) {
    // A rows 16 quad + lane (lanes 0-15), columns 32 half + [0, 32)
    float v[32];
    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + half * 32, v);
    if (lane < 16) {
      const int r = quad * 16 + lane;
      decay_row(v, GV, r, half * 32, true, GV.bt[r]);
#pragma unroll
      for (int i = 0; i < 32; i += 4)
        *reinterpret_cast<float4*>(Am + r * kLdF + half * 32 + i) =
            make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    }
    __syncthreads();
    solve_unit_lower(Am, Tm, Sm, tid, ST, [] { __syncthreads(); });
    // row r = tid / 4, 16-byte chunks 2 (tid % 4) + {0, 1}
    const int r = tid >> 2;
    unsigned char* dst = p.tiles + p.sq.template rec_t<Packed>(sqi, h, ci) * 8192;
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
      *reinterpret_cast<uint4*>(dst + sw_row_off(r, c8)) = pk;
    }
  } else if (tid == 0) {
    report_timeout();
    // nothing may still be writing this CTA's shared memory or TMEM at exit (bounded)
    if (!loaded) mbar_wait(bar_ld, 0, 10000);
    else mbar_wait(bar_mma, 0, 10000);
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, 64);
}

// ---------------------------------------------------------------- backward kernel
//
// Reverse chunk scan, one CTA per sequence.  The running state gradient is
// held transposed, dG = dH^T (dv x dk), fp32 in TMEM (128 columns; the dG_in
// product accumulates onto it) with a bf16 copy in shared memory as the MMA
// operand.  Each chunk's entry state G_in comes from the workspace (written
// by the forward kernel, in states mode or by the forward pass that filled a
// saved context), and so does its T tile (written by the solve kernel); the next chunk's tiles are requested as soon as each
// slot has been read for the last time.  With R = V - diag(e) K H_in,
// U = T diag(beta) R, T = (I + A)^-1:
//
//   MMA1  [K;Q] K^T, -G_in K^T, dG K^T  (one batch)
//                                  -> K K^T (kept in TMEM), Q K^T -> P,
//                                     R^T = V^T + (-G_in K^T) diag(e)
//   MMA   dO^T P                   -> dU^T = (dG K^T) diag(f) + dO^T P
//   MMA   U^T = (R^T diag beta) T^T,  dZ^T = dU^T T     (dZ = (I+A)^-T dU)
//   MMA   [dZ; dO] U^T             -> dA = -strict_lower(dZ U^T), dP = dO U^T
//   MMA   dG_in = eC dG + (e dO)^T Q - (e dR)^T K       (dR = diag(beta) dZ)
//   MMA   dQ^T = G_in^T (e dO)^T + K^T (dP o Gam)^T      (two accumulators)
//   MMA   dK^T = dG^T (U diag f)^T - G_in^T (e dR)^T + Q^T (dP o Gam)
//               + K^T (M + M^T),  M = diag(beta) dA o Gam
//
// dv = dR; dbeta_r = sum_c dZ_rc R_rc + sum_j dA_rj (K K^T o Gam)_rj.  dq, dk
// and dv are staged in shared memory and leave by TMA tensor stores.
//
// Log-gate gradient.  dgamma_r (the gradient of the chunk's cumulative log
// gate at row r) is the sum of the gate's appearances in the chunk, each
// taken from a full-precision chunk matrix the scan already holds:
//   e_r dO_r . (Q H_in)_r         q_r . (first accumulator of dQ)_r
//   + rowsum - colsum of Z = dP o P and of dA o A (A = beta K K^T o Gam)
//   - e_r dR_r . (K H_in)_r       K H_in from the -G_in K^T product
//   - s_r,  s_j = f_j u_j . (dG K^T)_j,
// and dg_t = sum_{s >= t in the chunk} dgamma_s + <dH_out, H_out>, the last
// term (from the chunk's own state update H_out = eC H_in + K^T diag(f) U) being
// eC <dH_out, H_in> + sum_j s_j.  The scalar gate's rescaling identity
// dgamma = q . dq - v . dv gives the same value but as a difference of two
// large, nearly equal sums once gates decay fast, where the bf16 rounding of
// dq and dv no longer cancels; the terms above carry no such cancellation.
// Keeping the sum inside the chunk avoids accumulating the rounding of
// thousands of terms.

constexpr int BT = 512;                  // backward threads (as the forward)
constexpr int kB_KQ = 0;                 // [Kh0 | Qh0 | Kh1 | Qh1]
constexpr int kB_ZO = 32768;             // [dZh0 | dOh0 | dZh1 | dOh1]
constexpr int kB_GI = 65536;             // G_in tile (K-major [c][d])
constexpr int kB_DG = 98304;             // dG tile (K-major [c][d])
constexpr int kB_V = 131072;             // [Vh0 | Vh1]
constexpr int kB_T = kB_V + 16384;       // T [r][j]; after the dZ product: M = beta dA o Gam
constexpr int kB_P = kB_T + 8192;        // P [r][j]; after dO^T P: dP o Gam
constexpr int kB_X = kB_P + 8192;        // three 16 KB slots, reused by phase
constexpr int kB_GATE = kB_X + 3 * 16384;  // gam, e, f, beta, er, ie, db1, db2, dlc [64] each, eC, fast
constexpr int kB_RED = kB_GATE + 9 * 256 + 16;  // reduction scratch, 1024 floats:
constexpr int kRedZ = 512;    //   [512, 768): rowsum(Z) partials [cg][r]
constexpr int kRedRow = 768;  //   [768, 832): the chunk's row-sum terms of dgamma
constexpr int kB_EC = kB_RED + 4096;
constexpr int kB_GRAW = kB_EC + 64;     // 2 x 128 raw g, beta (prefetch)
constexpr int kB_BAR = kB_GRAW + 2 * 512;
constexpr int kBwdSmemBytes = kB_BAR + 128 + 1024;
static_assert(kBwdSmemBytes <= 227 * 1024, "shared memory budget");

// TMEM columns of the backward kernel
constexpr uint32_t kBtKQ = 0, kBtR = 64, kBtX1 = 128, kBtX2 = 192, kBtU = 256, kBtZ = 320,
                   kBtG3 = 384;  // G3: 128 columns
// reused later: G4 -> X1 columns, dQ -> X2 columns, dK -> U columns

struct BwdParams {
  const float* g;
  const float* beta;
  const float* dht;
  const unsigned char* states;   // [B*H][N][32 KB]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dg;
  float* dbeta;
  float* dh0;
  const unsigned char* tiles;    // T of every chunk (8 KB per chunk record, from the solve kernel)
  int B, T, H, N;
  Seqs sq;
};

template <bool NoDelta, bool Packed>
__global__ void __launch_bounds__(BT, 1)
gdn_tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dq, const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv, BwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, cg = warp >> 2;
  const int row = quad * 32 + lane;
  const int bh = blockIdx.x, sq_s = bh / p.H, h = bh % p.H;
  int b = 0, tb = 0, slen = 0, NN = 0;  // batch row, first token, length, chunks (after the wait)

  float* gam = reinterpret_cast<float*>(sm + kB_GATE);
  float* ee = gam + 64;
  float* ff = ee + 64;
  float* bt = ff + 64;
  float* db1 = gam + 384;
  float* db2 = db1 + 64;
  float* dlc = db2 + 64;
  float* red = reinterpret_cast<float*>(sm + kB_RED);
  float* eC = reinterpret_cast<float*>(sm + kB_EC);
  const GateView GV{gam, ee, ff, bt, gam + 256, gam + 320, eC, gam + 576};
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + kB_BAR);
  uint64_t* bar_mma = bar_load + 1;
  uint64_t* bar_kq = bar_load + 2;  // K K^T, Q K^T done; later dO^T P done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_load + 3);
  // operand descriptors: every tile's is a base descriptor plus its offset
  const uint64_t dK0 = sw128_desc(smem_u32(sm), 16, 1024), dM0 = sw128_desc(smem_u32(sm), 16384, 1024);
  auto kdesc = [&](uint32_t off) { return desc_at(dK0, off); };  // K-major tiles
  auto mdesc = [&](uint32_t off) { return desc_at(dM0, off); };  // MN-major tiles

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    mbar_init(bar_kq, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmCols);
    tmem_relinquish();
  }
  cta_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lb = (uint32_t)(quad * 32) << 16;
  grid_dep_wait();  // the previous kernel's results (and its reads of what this one writes)
  grid_dep_launch();
  p.sq.get_t<Packed>(sq_s, b, tb, slen, NN);

  // The running state gradient dG (fp32) lives in TMEM columns kBtG3..+127
  // (row c = lane, column d); the dG_in product accumulates onto it.  This
  // thread's 32 columns: d in [32 cg, 32 cg + 32).
  const int g_region = cg >> 1, g_chunk0 = (cg & 1) * 4;
  const uint32_t t_dg = tmem + lb + kBtG3 + cg * 32;
  // bf16 copy of dG (the MMA operand)
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
  {
    float g[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) g[i] = p.dht ? p.dht[((size_t)bh * D + cg * 32 + i) * D + row] : 0.f;
    tmem_st32(t_dg, g);
    write_dg(g);
  }

  float* graw = reinterpret_cast<float*>(sm + kB_GRAW);
  auto load_gates = [&](int ci) {
    prefetch_gates(graw + (ci & 1) * 128, p.g, p.beta, (size_t)b * p.T + tb + ci * C,
                   min(C, slen - ci * C), p.H, h, lane);
  };
  // The gates of each chunk are computed by warp 1 near the end of the chunk
  // before it in the reverse scan, from g and beta prefetched one more chunk
  // ahead; the last chunk's here.
  if (warp == 0 && NN > 0) {
    load_gates(NN - 1);
    chunk_gates_raw(GV, graw + ((NN - 1) & 1) * 128, lane);
    if (NN > 1) load_gates(NN - 2);
  }

  uint32_t mma_phase = 0, load_phase = 0, kq_phase = 0;
  // dbeta and dg of a finished chunk are written by warps 4 and 5 while the
  // next chunk's first products run (their inputs, db1, db2, dlc and the
  // reduction scratch, are not rewritten before that chunk's E4)
  int pend_t0 = 0, pend_n = -1;
  auto flush_pending = [&]() {
    const size_t base = ((size_t)b * p.T + pend_t0) * p.H + h;
    if (warp == 5) {
      if (lane < pend_n) p.dbeta[base + (size_t)lane * p.H] = db1[lane] + db2[lane];
      if (lane + 32 < pend_n) p.dbeta[base + (size_t)(lane + 32) * p.H] = db1[lane + 32] + db2[lane + 32];
    } else if (warp == 4) {
      // dg_t = sum_{s >= t, s in chunk} dgamma_s + <dH_out, H_out>
      float carry = 0.f;
#pragma unroll
      for (int w = 0; w < BT / 32; ++w) carry += red[256 + w];
      float a0 = dlc[lane] + red[kRedRow + lane], a1 = dlc[lane + 32] + red[kRedRow + lane + 32];
      float s1 = a1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, s1, off);
        if (lane + off < 32) s1 += y;
      }
      const float tot1 = __shfl_sync(0xffffffffu, s1, 0);
      float s0 = a0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, s0, off);
        if (lane + off < 32) s0 += y;
      }
      s0 += tot1;
      if (lane < pend_n) p.dg[base + (size_t)lane * p.H] = carry + s0;
      if (lane + 32 < pend_n) p.dg[base + (size_t)(lane + 32) * p.H] = carry + s1;
    }
  };
  bool ok = true;
  auto mma_wait = [&]() {
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
  };

  // Tiles of chunk ci land on bar_load.  The loads for the next chunk of the
  // reverse scan are issued inside the current one as soon as each slot has
  // been read for the last time: V after the dv/dZ epilogue, K, dO, G_in and
  // T once the last products are done, Q after the q . dq sums.  The whole
  // chunk's byte count is announced with the first of them.
  constexpr uint32_t kChunkBytes = 8 * 8192 + 32768 + (NoDelta ? 0 : 8192);
  int inflight = -1;   // thread 0: chunk whose tiles are requested but not yet waited for
  int parts = 0;       // thread 0: how many of its three load groups are issued
  auto issue_v = [&](int cn) {
    const int tn = tb + cn * C;
    inflight = cn;
    parts = 1;
    mbar_arrive_expect_tx(bar_load, kChunkBytes);
    tma_load_4d(sm + kB_V, &tm_v, bar_load, 0, h, tn, b);
    tma_load_4d(sm + kB_V + 8192, &tm_v, bar_load, 64, h, tn, b);
  };
  auto issue_rest = [&](int cn) {
    const int tn = tb + cn * C;
    parts = 2;
    tma_load_4d(sm + kB_KQ + 0, &tm_k, bar_load, 0, h, tn, b);
    tma_load_4d(sm + kB_KQ + 16384, &tm_k, bar_load, 64, h, tn, b);
    tma_load_4d(sm + kB_ZO + 8192, &tm_do, bar_load, 0, h, tn, b);
    tma_load_4d(sm + kB_ZO + 24576, &tm_do, bar_load, 64, h, tn, b);
    bulk_load(sm + kB_GI, p.states + rec_bh<Packed>(p.sq, p.N, bh, sq_s, h, cn) * 32768, 32768, bar_load);
    if (!NoDelta) bulk_load(sm + kB_T, p.tiles + rec_bh<Packed>(p.sq, p.N, bh, sq_s, h, cn) * 8192, 8192, bar_load);
  };
  auto issue_q = [&](int cn) {
    const int tn = tb + cn * C;
    parts = 3;
    tma_load_4d(sm + kB_KQ + 8192, &tm_q, bar_load, 0, h, tn, b);
    tma_load_4d(sm + kB_KQ + 24576, &tm_q, bar_load, 64, h, tn, b);
  };
  if (tid == 0 && NN > 0) {
    issue_v(NN - 1);
    issue_rest(NN - 1);
    issue_q(NN - 1);
  }

  for (int ci = NN - 1; ci >= 0 && ok; --ci) {
    const int t0 = tb + ci * C, n = min(C, slen - ci * C);
    const bool rowwise = Packed && n < C;  // a packed sequence's partial last chunk
    fence_async_shared();  // the dG tile written last chunk, for MMA1 (after the barrier below)
    ok = __syncthreads_and(mbar_wait(bar_load, load_phase));
    if (!ok) break;
    load_phase ^= 1;
    inflight = -1;
    if (rowwise) {
      // rows past the sequence hold the next one's dO: zero them, so that no
      // product carries them into this sequence's gradients (the gates of
      // those rows are already masked to g = 0, beta = 0)
      for (int i = tid; i < (C - n) * 16; i += BT) {
        const int r = n + (i >> 4), hh = (i >> 3) & 1, c8 = i & 7;
        *reinterpret_cast<uint4*>(sm + kB_ZO + hh * 16384 + 8192 + r * 128 + c8 * 16) =
            make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (NoDelta) {
      // T = I (the tile slot is rewritten later in the chunk): thread tid writes
      // the 16-byte chunk tid % 8 of row tid / 8
      const int r = tid >> 3, c8 = tid & 7;
      uint4 pk = make_uint4(0u, 0u, 0u, 0u);
      if ((r >> 3) == c8) reinterpret_cast<__nv_bfloat16*>(&pk)[r & 7] = __float2bfloat16_rn(1.f);
      *reinterpret_cast<uint4*>(sm + kB_T + sw_row_off(r, c8)) = pk;
    }
    // ---- MMA1: [K;Q] K^T, committed on its own so that the P epilogue runs
    // while the tensor cores go on with -G_in K^T (not formed without the
    // delta rule) and dG K^T
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      const uint32_t idn = idesc_bf16(128, 64, false, false, true);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        mma_bf16(tmem + kBtKQ, kdesc(kB_KQ + off), kdesc(kB_KQ + off), id, ks > 0);
      }
      mma_commit(bar_kq);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        if (!NoDelta)
          mma_bf16(tmem + kBtR, kdesc(kB_GI + off), kdesc(kB_KQ + off), idn, ks > 0);
        mma_bf16(tmem + kBtX1, kdesc(kB_DG + off), kdesc(kB_KQ + off), id, ks > 0);
      }
      mma_commit(bar_mma);
    }
    if (pend_n >= 0) flush_pending();  // the chunk before, in warps 4 and 5
    // P = lower(Q K^T o Gam) from TMEM lanes 64-127 (warps of the upper two
    // lane quarters; the issuing thread is in the first)
    {
      bool okp = true;
      if (row >= 64) {
        okp = mbar_wait(bar_kq, kq_phase);
        tc_fence_after();
        if (okp) {
          const int r = row - 64;
          float v[16];
          tmem_ld16(tmem + lb + kBtKQ + cg * 16, v);
          decay_row(v, GV, r, cg * 16, false, 1.f);
          store_chunks(sm + kB_P, r, cg * 2, v, 2);
        }
      }
      kq_phase ^= 1;
      fence_async_shared();
      tc_fence_before();
      ok = __syncthreads_and(okp);
      tc_fence_after();
      if (!ok) break;
    }
    // ---- dO^T P
    if (tid == 0) {
      const uint32_t idmm = idesc_bf16(128, 64, true, true);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtX2, mdesc(kB_ZO + 8192 + ks * 2048),
                 mdesc(kB_P + ks * 2048), idmm, ks > 0);
      mma_commit(bar_kq);
      bulk_wait_read_all();  // the previous chunk's dq / dk staging (X0, X1) has been read
    }
    // This commit arrives once every product issued so far is done, the rest of
    // MMA1 included: its own phase on bar_mma is passed over (a later wait on
    // bar_mma targets the newest phase, which completes after it).
    ok = __syncthreads_and(mbar_wait(bar_kq, kq_phase));
    kq_phase ^= 1;
    mma_phase ^= 1;
    tc_fence_after();
    if (!ok) break;
    // ---- E3: beta R^T -> X0, dU^T -> X1  (this thread: row c, columns 16 cg + i)
    {
      float a[16], x[16];
      tmem_ld16(tmem + lb + kBtR + cg * 16, a);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = cg * 16 + i;
        const float kh = NoDelta ? 0.f : ee[r] * a[i];
        a[i] = bt[r] * (tile_elem(sm + kB_V + (row >> 6) * 8192, r, row & 63) + kh);
      }
      store_chunks(sm + kB_X, row, cg * 2, a, 2);
      tmem_ld16(tmem + lb + kBtX1 + cg * 16, a);
      tmem_ld16(tmem + lb + kBtX2 + cg * 16, x);
#pragma unroll
      for (int i = 0; i < 16; ++i) a[i] = ff[cg * 16 + i] * a[i] + x[i];
      store_chunks(sm + kB_X + 16384, row, cg * 2, a, 2);
    }
    fence_async_shared();
    cta_sync();
    // ---- U^T = (beta R^T) T^T,  dZ^T = dU^T T
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      const uint32_t idm = idesc_bf16(128, 64, false, true);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tmem + kBtU, kdesc(kB_X + ks * 32), kdesc(kB_T + ks * 32), id,
                 ks > 0);
        mma_bf16(tmem + kBtZ, kdesc(kB_X + 16384 + ks * 32), mdesc(kB_T + ks * 2048),
                 idm, ks > 0);
      }
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // ---- E4: U^T -> X0, (U diag f)^T -> X2, e dR^T -> X1, dZ rows -> ZO, dv, dbeta part 1
    float acc[16];  // this thread's terms of the log-gate gradient, columns 16 cg + i
    {
      // <dH_out, H_out> of this chunk, with H_out = eC H_in + K^T diag(f) U its
      // state update: eC <dG, G_in> + sum_{c,j} (U diag f)^T_cj (dG K^T)_cj
      float cdot = 0.f;
      {
        float g[32];
        tmem_ld32(t_dg, g);  // dG_out
        const unsigned char* tile = sm + kB_GI + g_region * 16384;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 pk = *reinterpret_cast<const uint4*>(tile + sw_row_off(row, g_chunk0 + k));
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f2 = __bfloat1622float2(h2[i]);
            cdot = fmaf(g[k * 8 + 2 * i], f2.x, cdot);
            cdot = fmaf(g[k * 8 + 2 * i + 1], f2.y, cdot);
          }
        }
        const float ec = *eC;
        cdot *= ec;
        // dG <- eC dG; the dG_in product of this chunk accumulates onto it
#pragma unroll
        for (int i = 0; i < 32; ++i) g[i] *= ec;
        tmem_st32(t_dg, g);
      }
      float u[16];
      tmem_ld16(tmem + lb + kBtU + cg * 16, u);
      store_chunks(sm + kB_X, row, cg * 2, u, 2);
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] *= ff[cg * 16 + i];
      store_chunks(sm + kB_X + 32768, row, cg * 2, u, 2);
      {
        // s_j = f_j u_j . (dG K^T)_j enters dgamma_j with a minus sign and the
        // chunk-end carry with a plus sign
        float x1[16];
        tmem_ld16(tmem + lb + kBtX1 + cg * 16, x1);  // dG K^T, row c, columns j
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float sj = u[i] * x1[i];
          cdot += sj;
          acc[i] = -sj;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) cdot += __shfl_xor_sync(0xffffffffu, cdot, off);
      if (lane == 0) red[256 + warp] = cdot;  // summed by warp 0 for dg
      float z[16], rr[16];
      tmem_ld16(tmem + lb + kBtZ + cg * 16, z);
      tmem_ld16(tmem + lb + kBtR + cg * 16, rr);
      if (NoDelta) {
#pragma unroll
        for (int i = 0; i < 16; ++i) rr[i] = 0.f;  // R = V
      }
      const int half = row >> 6, cc = row & 63;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = cg * 16 + i;
        const float vr = tile_elem(sm + kB_V + half * 8192, r, cc);
        const float dr = bt[r] * z[i];
        acc[i] = fmaf(ee[r] * dr, rr[i], acc[i]);  // -e_r dR_rc (K H_in)_rc  (rr = -(K H_in)^T)
        rr[i] = z[i] * (vr + ee[r] * rr[i]);      // dZ_rc R_rc
        z[i] = ee[r] * dr;
      }
      // dv = dR (T and P have been read for the last time) and the dZ rows of the
      // [dZ; dO] operand, token-major: transposed stores of this warp's block
      const uint32_t tz = tmem + lb + kBtZ + cg * 16;
      stage_tmem_block(sm + kB_T, 8192, tz, quad * 32, cg * 16, [&](int r, float zz) { return bt[r] * zz; });
      stage_tmem_block(sm + kB_ZO, 16384, tz, quad * 32, cg * 16, [](int, float zz) { return zz; });
      store_chunks(sm + kB_X + 16384, row, cg * 2, z, 2);
      cta_sum_rows16(rr, red, db1);
    }
    fence_async_shared();
    cta_sync();
    // ---- G4: [dZ; dO] U^T  (lanes 0-63: dZ U^T, lanes 64-127: dO U^T)
    if (rowwise)
      store_rows_bf16(sm + kB_T, p.dv + (((size_t)b * p.T + t0) * p.H + h) * D, (size_t)p.H * D, n, tid,
                      BT);
    if (tid == 0) {
      // dv: TMA store of the staged tile (rows past T are not written)
      if (!rowwise) {
        tma_store_4d(&tm_dv, sm + kB_T, 0, h, t0, b);
        tma_store_4d(&tm_dv, sm + kB_T + 8192, 64, h, t0, b);
      }
      bulk_commit_group();
      if (ci > 0) issue_v(ci - 1);  // V has been read for the last time
      const uint32_t id = idesc_bf16(128, 64, false, true);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtX1, kdesc(kB_ZO + (ks / 4) * 16384 + (ks % 4) * 32),
                 mdesc(kB_X + ks * 2048), id, ks > 0);
      mma_commit(bar_mma);
      bulk_wait_read_all();  // the staged dv is read before M and dP o Gam overwrite it
    }
    mma_wait();
    if (!ok) break;
    {
      float x[16];
      tmem_ld16(tmem + lb + kBtX1 + cg * 16, x);
      if (row < 64) {
        // dA = -strict_lower(dZ U^T); dbeta part 2: sum_j dA_rj (K K^T o Gam)_rj;
        // M = beta dA o Gam
        const int r = row;
        float kk[16];
        tmem_ld16(tmem + lb + kBtKQ + cg * 16, kk);
        const float br = bt[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = NoDelta ? 0.f : -x[i];  // no A without the delta rule
        decay_row(x, GV, r, cg * 16, true, 1.f);   // x = dA o Gam
        float s2 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float t = x[i] * kk[i];
          s2 += t;
          acc[i] = fmaf(-br, t, acc[i]);  // -colsum(dA o A)
          x[i] *= br;
        }
        red[cg * 64 + r] = s2;             // rowsum(dA o A) = beta_r * (sum over cg)
        store_chunks(sm + kB_T, r, cg * 2, x, 2);
      } else {
        // Z = dP o P with P = Q K^T o Gam (Q K^T still in these TMEM lanes)
        const int r = row - 64;
        float qk[16];
        tmem_ld16(tmem + lb + kBtKQ + cg * 16, qk);
        decay_row(x, GV, r, cg * 16, false, 1.f);  // x = dP o Gam
        float sz = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float t = x[i] * qk[i];
          sz += t;
          acc[i] -= t;                     // -colsum(Z)
        }
        red[kRedZ + cg * 64 + r] = sz;     // rowsum(Z) partial
        store_chunks(sm + kB_P, r, cg * 2, x, 2);
      }
    }
    // scale dO rows by e in place (dO is done as an operand of dO^T P and G4)
    for (int i = tid; i < 2 * 64 * 8; i += BT) {
      const int half = i / 512, r = (i / 8) % 64, c8 = i % 8;
      uint4* ptr = reinterpret_cast<uint4*>(sm + kB_ZO + half * 16384 + 8192 + r * 128 + c8 * 16);
      uint4 val = *ptr;
      __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&val);
      const float e = ee[r];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float2 f2 = __bfloat1622float2(h2[k]);
        h2[k] = __floats2bfloat162_rn(f2.x * e, f2.y * e);
      }
      *ptr = val;
    }
    fence_async_shared();
    cta_sync();
    if (tid < 64) {
      const float s2 = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
      db2[tid] = s2;
      // rowsum(dA o A) + rowsum(Z) of this chunk's log-gate gradient
      red[kRedRow + tid] = bt[tid] * s2 + red[kRedZ + tid] + red[kRedZ + 64 + tid] +
                           red[kRedZ + 128 + tid] + red[kRedZ + 192 + tid];
    }
    // ---- dG_in part, dQ^T, dK^T
    if (tid == 0) {
      // G3 = (e dO)^T Q - (e dR)^T K   [c x d]
      const uint32_t idg = idesc_bf16(128, 128, true, true);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtG3, mdesc(kB_ZO + 8192 + ks * 2048),
                 mdesc(kB_KQ + 8192 + ks * 2048), idg, 1);
      const uint32_t idgn = idesc_bf16(128, 128, false, true, true);
      #pragma unroll
      for (int ks = 0; ks < (NoDelta ? 0 : 4); ++ks)
        mma_bf16(tmem + kBtG3, kdesc(kB_X + 16384 + ks * 32), mdesc(kB_KQ + ks * 2048),
                 idgn, 1);
      // dQ^T = G_in^T (e dO)^T + K^T (dP o Gam)^T   [d x r], the two terms in
      // separate accumulators (R columns, X2 columns): q . (first term) is the
      // state's part of the log-gate gradient
      const uint32_t idq = idesc_bf16(128, 64, true, false);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtR, mdesc(kB_GI + ks * 2048),
                 kdesc(kB_ZO + 8192 + (ks / 4) * 16384 + (ks % 4) * 32), idq, ks > 0);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtX2, mdesc(kB_KQ + ks * 2048), kdesc(kB_P + ks * 32),
                 idq, ks > 0);
      // dK^T  [d x j] -> U columns
      const uint32_t idmm = idesc_bf16(128, 64, true, true);
      const uint32_t idmmn = idesc_bf16(128, 64, true, true, true);
      #pragma unroll
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtU, mdesc(kB_DG + ks * 2048), mdesc(kB_X + 32768 + ks * 2048),
                 idmm, ks > 0);
      const int nd = NoDelta ? 0 : 1;  // the R- and A-terms vanish without the delta rule
      #pragma unroll
      for (int ks = 0; ks < 8 * nd; ++ks)
        mma_bf16(tmem + kBtU, mdesc(kB_GI + ks * 2048), mdesc(kB_X + 16384 + ks * 2048),
                 idmmn, 1);
      #pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtU, mdesc(kB_KQ + 8192 + ks * 2048),
                 mdesc(kB_P + ks * 2048), idmm, 1);
      #pragma unroll
      for (int ks = 0; ks < 4 * nd; ++ks)
        mma_bf16(tmem + kBtU, mdesc(kB_KQ + ks * 2048), kdesc(kB_T + ks * 32),
                 idq, 1);
      #pragma unroll
      for (int ks = 0; ks < 4 * nd; ++ks)
        mma_bf16(tmem + kBtU, mdesc(kB_KQ + ks * 2048), mdesc(kB_T + ks * 2048),
                 idmm, 1);
      mma_commit(bar_mma);
    }
    if (warp == 1 && ci > 0) {
      // gates of the next chunk of the reverse scan, while the products run
      // (nothing from here on in this chunk reads them)
      chunk_gates_raw(GV, graw + ((ci - 1) & 1) * 128, lane);
      if (ci > 1) load_gates(ci - 2);
    }
    // this thread's Q values for the q . dq sums (bf16 pairs), read while the
    // products run so that Q can be reloaded as soon as they are done
    __nv_bfloat162 qv[8];
    {
      const unsigned char* qt = sm + kB_KQ + (row >> 6) * 16384 + 8192;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = cg * 16 + 2 * i, cc = row & 63;
        qv[i].x = *reinterpret_cast<const __nv_bfloat16*>(qt + sw_row_off(r, cc >> 3) + (cc & 7) * 2);
        qv[i].y = *reinterpret_cast<const __nv_bfloat16*>(qt + sw_row_off(r + 1, cc >> 3) + (cc & 7) * 2);
      }
    }
    fence_async_shared();  // these reads come before the TMA that overwrites Q
    mma_wait();
    if (!ok) break;
    // ---- E6: dG update, dq (+ q.dq), dk, dbeta, dg
    // K, Q, dO, G_in and T have been read for the last time
    if (tid == 0 && ci > 0) {
      issue_rest(ci - 1);
      issue_q(ci - 1);
    }
    {
      {
        float g[32];
        tmem_ld32(t_dg, g);  // dG_in = eC dG_out + (e dO)^T Q - (e dR)^T K
        write_dg(g);         // the products that read the old copy are done
      }
      float x[16];
      tmem_ld16(tmem + lb + kBtR + cg * 16, x);  // dQ^T state term, row d = row, columns r = 16 cg + i
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 q2 = __bfloat1622float2(qv[i / 2]);
        acc[i] = fmaf((i & 1) ? q2.y : q2.x, x[i], acc[i]);  // e_r dO_r . (Q H_in)_r
      }
      // dq = both dQ^T terms (X0 is free once the products are done), dk (X1):
      // transposed stores of this warp's blocks
      stage_tmem_block(sm + kB_X, 8192, tmem + lb + kBtR + cg * 16, quad * 32, cg * 16,
                       [](int, float q) { return q; }, tmem + lb + kBtX2 + cg * 16);
      stage_tmem_block(sm + kB_X + 16384, 8192, tmem + lb + kBtU + cg * 16, quad * 32, cg * 16,
                       [](int, float q) { return q; });
    }
    fence_async_shared();
    cta_sum_rows16(acc, red, dlc);  // (its barriers also publish the staged dq, dk)
    if (rowwise) {
      const size_t o0 = (((size_t)b * p.T + t0) * p.H + h) * D;
      store_rows_bf16(sm + kB_X, p.dq + o0, (size_t)p.H * D, n, tid, BT);
      store_rows_bf16(sm + kB_X + 16384, p.dk + o0, (size_t)p.H * D, n, tid, BT);
    } else if (tid == 0) {
      tma_store_4d(&tm_dq, sm + kB_X, 0, h, t0, b);
      tma_store_4d(&tm_dq, sm + kB_X + 8192, 64, h, t0, b);
      tma_store_4d(&tm_dk, sm + kB_X + 16384, 0, h, t0, b);
      tma_store_4d(&tm_dk, sm + kB_X + 24576, 64, h, t0, b);
      bulk_commit_group();
    }
    pend_t0 = t0;
    pend_n = n;
  }

  if (ok && pend_n >= 0) flush_pending();  // the last chunk of the reverse scan
  if (!ok) {
    if (tid == 0) {
      report_timeout();
      // let the tile loads still in flight land before the CTA exits (bounded)
      if (inflight >= 0) {
        if (parts < 2) issue_rest(inflight);
        if (parts < 3) issue_q(inflight);
        mbar_wait(bar_load, load_phase, 10000);
      }
    }
  } else if (p.dh0) {
    float g[32];
    tmem_ld32(t_dg, g);
#pragma unroll
    for (int i = 0; i < 32; ++i) p.dh0[((size_t)bh * D + cg * 32 + i) * D + row] = g[i];
  }
  if (tid == 0) bulk_wait_all();  // the TMA stores of dq, dk, dv are complete
  cp_async_wait_all();  // no gate prefetch may still be writing shared memory at exit
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

// ---------------------------------------------------------------- wait self-test
//
// One CTA that takes the scan kernels' timeout branch on purpose: it sets up
// an mbarrier and TMEM as they do, then waits on the barrier with a bounded
// number of polls while nothing can arrive on it (no thread arrives and no
// copy or MMA is issued), so the wait runs out.  The CTA then records
// GDN_ERR_DEVICE_TIMEOUT in the device status word, frees its TMEM and
// returns -- the path a real timeout takes, with nothing in flight.

__global__ void __launch_bounds__(128, 1) gdn_wait_selftest_kernel(uint32_t max_tries) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int warp = threadIdx.x / 32;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&tmem_slot, 32);
    tmem_relinquish();
  }
  cta_sync();
  const uint32_t tmem = tmem_slot;
  const bool ok = __syncthreads_and(mbar_wait(&bar, 0, max_tries));
  if (!ok && threadIdx.x == 0) report_timeout();
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, 32);
}

// ---------------------------------------------------------------- packed sequences
//
// One CTA: checks that cu_seqlens rises from 0 to T without decreasing, then
// writes each sequence's first global chunk, chunk_off[s] = sum of
// ceil(len / C) over the sequences before it (chunk_off[nseq] = all chunks).
// Invalid offsets are recorded as GDN_ERR_SEQLENS and give zero chunks.

constexpr int kSetupThreads = 1024;

__global__ void __launch_bounds__(kSetupThreads)
gdn_setup_seqlens_kernel(const int* cu, int nseq, int T, int Cc, int* chunk_off) {
  __shared__ int bad, carry;
  __shared__ int warp_sum[kSetupThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    bad = (cu[0] != 0 || cu[nseq] != T) ? 1 : 0;
    carry = 0;
  }
  __syncthreads();
  for (int s = tid; s < nseq; s += kSetupThreads)
    if (cu[s + 1] < cu[s]) bad = 1;
  __syncthreads();
  for (int base = 0; base < nseq; base += kSetupThreads) {
    const int s = base + tid;
    const int c = (!bad && s < nseq) ? (cu[s + 1] - cu[s] + Cc - 1) / Cc : 0;
    int x = c;  // inclusive scan within the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) warp_sum[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sum[lane];
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = carry + (warp > 0 ? warp_sum[warp - 1] : 0) + x - c;
    if (s < nseq) chunk_off[s] = before;
    __syncthreads();
    if (tid == kSetupThreads - 1) carry = before + c;
    __syncthreads();
  }
  if (tid == 0) {
    chunk_off[nseq] = carry;
    if (bad) atomicExch(&g_file_status, GDN_ERR_SEQLENS);
  }
}

// ---------------------------------------------------------------- host side

// T tiles of every chunk into `tiles` ([B*H][N][8 KB])
cudaError_t launch_solve(const Problem& p, cudaStream_t s, unsigned char* tiles) {
  CUtensorMap mk;
  cudaError_t e;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  SolveParams sp{p.g, p.beta, tiles, p.B, p.T, p.H, p.N, Seqs::of(p), p.nseq};
  auto kern = p.cu_seqlens ? gdn_tc_solve_kernel<true> : gdn_tc_solve_kernel<false>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSolveSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  e = launch_overlapped(kern, (unsigned)(max_chunks(p) * p.H), ST,
                        kSolveSmemBytes, s, mk, sp);
  prof_after(s, kTcSolve);
  return e;
}

// One launch of the forward kernel.  Without segments: the whole forward
// (want_out) or the states pass (states != nullptr).  With seg_chunks > 0:
// one pass of the segmented forward (h0 / ht per segment).
struct FwdLaunch {
  bool want_out = false;
  __nv_bfloat16* states = nullptr;
  const float* h0 = nullptr;
  float* ht = nullptr;
  int seg_chunks = 0, v_zero = 0, h0_identity = 0;
  int kernel_id = kTcFwd;
};

cudaError_t launch_fwd(const Problem& p, cudaStream_t s, const unsigned char* tiles,
                       const FwdLaunch& f) {
  CUtensorMap mq, mk, mv, mo;
  cudaError_t e;
  if ((e = make_token_map(&mq, p.q, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mv, p.v, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mo, f.want_out ? p.o : p.q, p)) != cudaSuccess) return e;  // unused without output
  FwdParams fp{p.g, p.beta, f.h0, f.want_out ? static_cast<__nv_bfloat16*>(p.o) : nullptr,
               f.ht, f.states, tiles, p.B, p.T, p.H, p.N, Seqs::of(p), f.seg_chunks, f.v_zero,
               f.h0_identity};
  // the Mamba2 mixer (no delta rule) is a separate instance: T = I, no W products
  auto kern = p.cu_seqlens ? (p.no_delta ? gdn_tc_fwd_kernel<true, true> : gdn_tc_fwd_kernel<false, true>)
                           : (p.no_delta ? gdn_tc_fwd_kernel<true, false> : gdn_tc_fwd_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int nseg = f.seg_chunks ? (p.N + f.seg_chunks - 1) / f.seg_chunks : 1;
  prof_before(s);
  e = launch_overlapped(kern, (unsigned)((size_t)num_seqs(p) * p.H * nseg), FT, kSmemBytes, s, mq, mk,
                        mv, mo, fp);
  prof_after(s, f.kernel_id);
  return e;
}

// ---------------------------------------------------------------- segmented forward
//
// A sequence's state map over a run of chunks is affine, H_out = M H_in + N:
// M is the run with V = 0 started from H = I, N the run started from H = 0.
// With few sequences and many chunks (a long context), the forward splits
// each sequence into segments so that every SM has work: pass 1 computes M
// and N of every segment in parallel, the combine kernel chains
// H_in(s+1) = M_s H_in(s) + N_s in fp32 per sequence, and pass 2 reruns every
// segment from its entry state to produce the output.  About three times the
// arithmetic of the plain forward, spread over B*H*nseg CTAs instead of B*H.

constexpr int kCombineThreads = 256;
constexpr int kCombineSplit = 8;               // CTAs per sequence, each a block of H's columns
constexpr int kCombineCols = D / kCombineSplit;  // 16 columns of H (dv) per CTA
constexpr int kCombineLdM = D + 1;             // M row stride in shared memory (no bank conflicts)
constexpr int kCombineSmem = (D * kCombineLdM + D * kCombineCols) * 4;  // M, then the H block, fp32

// H_in(s + 1) = M_s H_in(s) + N_s acts on each column of H on its own, so
// the columns are split over kCombineSplit CTAs per sequence.  Thread t
// owns row d = t / 2 and columns 8 (t % 2) + [0, 8) of its CTA's block.
__global__ void __launch_bounds__(kCombineThreads)
gdn_tc_combine_kernel(const float* M, const float* Nl, const float* h0, float* Hin, float* ht,
                      int nseg) {
  extern __shared__ float csm[];
  float* Ms = csm;                       // [dk][dk], row stride kCombineLdM
  float* Hs = csm + D * kCombineLdM;     // [dk][kCombineCols]
  const int t = threadIdx.x, bh = blockIdx.x / kCombineSplit;
  const int c0 = (blockIdx.x % kCombineSplit) * kCombineCols;  // first column of H
  const int d = t >> 1, e0 = (t & 1) * 8;
  for (int i = t; i < D * kCombineCols; i += kCombineThreads) {
    const int r = i / kCombineCols, c = i % kCombineCols;
    Hs[i] = h0 ? h0[((size_t)bh * D + r) * D + c0 + c] : 0.f;
  }
  __syncthreads();
  for (int sgi = 0; sgi < nseg; ++sgi) {
    const size_t base = ((size_t)bh * nseg + sgi) * D * D;
    for (int i = t; i < D * kCombineCols; i += kCombineThreads) {
      const int r = i / kCombineCols, c = i % kCombineCols;
      Hin[base + (size_t)r * D + c0 + c] = Hs[i];
    }
    for (int i = t; i < D * D / 4; i += kCombineThreads) {
      const float4 m4 = reinterpret_cast<const float4*>(M + base)[i];
      const int r = (4 * i) / D, c = (4 * i) % D;
      float* dst = Ms + r * kCombineLdM + c;
      dst[0] = m4.x;
      dst[1] = m4.y;
      dst[2] = m4.z;
      dst[3] = m4.w;
    }
    float acc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = Nl[base + (size_t)d * D + c0 + e0 + j];
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < D; ++k) {
      const float m = Ms[d * kCombineLdM + k];
      const float4 h_lo = *reinterpret_cast<const float4*>(Hs + k * kCombineCols + e0);
      const float4 h_hi = *reinterpret_cast<const float4*>(Hs + k * kCombineCols + e0 + 4);
      acc[0] = fmaf(m, h_lo.x, acc[0]);
      acc[1] = fmaf(m, h_lo.y, acc[1]);
      acc[2] = fmaf(m, h_lo.z, acc[2]);
      acc[3] = fmaf(m, h_lo.w, acc[3]);
      acc[4] = fmaf(m, h_hi.x, acc[4]);
      acc[5] = fmaf(m, h_hi.y, acc[5]);
      acc[6] = fmaf(m, h_hi.z, acc[6]);
      acc[7] = fmaf(m, h_hi.w, acc[7]);
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 8; ++j) Hs[d * kCombineCols + e0 + j] = acc[j];
    __syncthreads();
  }
  if (ht)
    for (int i = t; i < D * kCombineCols; i += kCombineThreads) {
      const int r = i / kCombineCols, c = i % kCombineCols;
      ht[((size_t)bh * D + r) * D + c0 + c] = Hs[i];
    }
}

// Chunks per segment of the forward pass, or 0 for no segments.  A pass over
// nseg segments per sequence takes about waves x (chunks per segment) chunk
// times, waves = ceil(seqs nseg / SMs) with one CTA per SM; the segmented
// forward runs three such passes (transitions, local states, outputs).  The
// count with the least time is taken (the smallest of equals), and segments
// are used only when three passes beat one unsegmented pass by a third.
// Segments are at least 32 chunks long.
int fwd_seg_chunks(const Problem& p) {
  if (p.no_delta || p.cu_seqlens) return 0;  // segments: GDN batches only
  const long seqs = (long)p.B * p.H;
  const long sms = sm_count();
  if (seqs <= 0 || sms <= 0 || p.N < 128) return 0;
  auto waves = [&](long ctas) { return (ctas + sms - 1) / sms; };
  const long plain = waves(seqs) * p.N;
  long best = 0, best_cost = 0;
  for (long nseg = 2; nseg <= p.N / 32; ++nseg) {
    const long cost = 3 * waves(seqs * nseg) * ((p.N + nseg - 1) / nseg);
    if (best == 0 || cost < best_cost) best = nseg, best_cost = cost;
  }
  if (best == 0 || 3 * best_cost > 2 * plain) return 0;
  return (int)((p.N + best - 1) / best);
}

size_t seg_state_bytes(const Problem& p, int seg_chunks) {
  const int nseg = (p.N + seg_chunks - 1) / seg_chunks;
  return align_up((size_t)p.B * p.H * nseg * D * D * 4, 256);
}

}  // namespace

cudaError_t setup_seqlens(const Problem& p, int* chunk_off, cudaStream_t s) {
  prof_before(s);
  gdn_setup_seqlens_kernel<<<1, kSetupThreads, 0, s>>>(p.cu_seqlens, p.nseq, p.T, p.C, chunk_off);
  prof_after(s, kSeqSetup);
  return cudaGetLastError();
}

cudaError_t wait_selftest(int max_tries, cudaStream_t s) {
  gdn_wait_selftest_kernel<<<1, 128, 0, s>>>((uint32_t)max_tries);
  return cudaGetLastError();
}

bool tc_supported(const Problem& p) {
  return p.bf16 && !p.kda && p.dk == D && p.dv == D && p.C == C;
}

size_t tiles_bytes(const Problem& p) { return align_up((size_t)max_chunks(p) * p.H * 8192, 256); }
size_t states_bytes(const Problem& p) { return align_up((size_t)max_chunks(p) * p.H * 32768, 256); }

size_t seg_scratch_bytes(const Problem& p) {
  const int sc = fwd_seg_chunks(p);
  return sc ? 3 * seg_state_bytes(p, sc) : 0;
}

// Workspace of the tensor-core forward pass: the T tile of every chunk; with
// segments also M, N and the entry state of every segment (fp32, dk x dv).
size_t tc_fwd_workspace(const Problem& p) { return tiles_bytes(p) + seg_scratch_bytes(p); }

// Workspace of the tensor-core backward pass: the bf16 entry state of every
// chunk in MMA-operand layout (32 KB each), then the T tile of every chunk.
size_t tc_bwd_workspace(const Problem& p) { return states_bytes(p) + tiles_bytes(p); }

// Saved context: the backward pass's workspace as the forward pass leaves it
// (entry states, then T tiles), then the forward's segment scratch.
size_t tc_ctx_bytes(const Problem& p) { return tc_bwd_workspace(p) + seg_scratch_bytes(p); }

// With save, the workspace is a saved context: the output pass also writes
// every chunk's bf16 entry state in front of the T tiles, where the backward
// pass of the same inputs finds both.
cudaError_t tc_fwd(const Problem& p, cudaStream_t s, bool save) {
  unsigned char* ws = static_cast<unsigned char*>(p.ws);
  __nv_bfloat16* states = save ? reinterpret_cast<__nv_bfloat16*>(ws) : nullptr;
  unsigned char* tiles = save ? ws + states_bytes(p) : ws;
  cudaError_t e = p.no_delta ? cudaSuccess : launch_solve(p, s, tiles);  // T = I without the delta rule
  if (e != cudaSuccess) return e;
  const int sc = fwd_seg_chunks(p);
  if (!sc) {
    FwdLaunch f;
    f.want_out = true;
    f.states = states;
    f.h0 = p.h0;
    f.ht = p.ht;
    return launch_fwd(p, s, tiles, f);
  }
  const int nseg = (p.N + sc - 1) / sc;
  const size_t sb = seg_state_bytes(p, sc);
  float* Mt = reinterpret_cast<float*>(tiles + tiles_bytes(p));
  float* Nl = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(Mt) + sb);
  float* Hin = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(Nl) + sb);
  FwdLaunch m;  // transitions: V = 0 from H = I
  m.ht = Mt;
  m.seg_chunks = sc;
  m.v_zero = 1;
  m.h0_identity = 1;
  m.kernel_id = kTcSegment;
  if ((e = launch_fwd(p, s, tiles, m)) != cudaSuccess) return e;
  FwdLaunch n;  // local states from H = 0
  n.ht = Nl;
  n.seg_chunks = sc;
  n.kernel_id = kTcSegment;
  if ((e = launch_fwd(p, s, tiles, n)) != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gdn_tc_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kCombineSmem);
  if (e != cudaSuccess) return e;
  prof_before(s);
  gdn_tc_combine_kernel<<<p.B * p.H * kCombineSplit, kCombineThreads, kCombineSmem, s>>>(Mt, Nl, p.h0, Hin, p.ht,
                                                                          nseg);
  prof_after(s, kTcCombine);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  FwdLaunch o;  // outputs from every segment's entry state
  o.want_out = true;
  o.states = states;
  o.h0 = Hin;
  o.seg_chunks = sc;
  return launch_fwd(p, s, tiles, o);
}

// With saved, the workspace is a context filled by tc_fwd(save) on the same
// inputs: the solve and the states pass are not run again.
cudaError_t tc_bwd(const Problem& p, cudaStream_t s, bool saved) {
  unsigned char* ws = static_cast<unsigned char*>(p.ws);
  __nv_bfloat16* states = reinterpret_cast<__nv_bfloat16*>(ws);
  unsigned char* tiles = ws + states_bytes(p);
  cudaError_t e;
  if (!saved) {
    if (!p.no_delta && (e = launch_solve(p, s, tiles)) != cudaSuccess) return e;
    FwdLaunch st;
    st.states = states;
    st.h0 = p.h0;
    st.kernel_id = kTcStates;
    if ((e = launch_fwd(p, s, tiles, st)) != cudaSuccess) return e;
  }
  CUtensorMap mq, mk, mv, mdo, mdq, mdk, mdv;
  if ((e = make_token_map(&mq, p.q, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mv, p.v, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdo, p.do_, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdq, p.dq, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdk, p.dk_, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdv, p.dv_, p)) != cudaSuccess) return e;
  BwdParams bp{p.g, p.beta, p.dht,
               reinterpret_cast<const unsigned char*>(states), static_cast<__nv_bfloat16*>(p.dq),
               static_cast<__nv_bfloat16*>(p.dk_), static_cast<__nv_bfloat16*>(p.dv_), p.dg, p.dbeta,
               p.dh0, tiles, p.B, p.T, p.H, p.N, Seqs::of(p)};
  auto kern = p.cu_seqlens ? (p.no_delta ? gdn_tc_bwd_kernel<true, true> : gdn_tc_bwd_kernel<false, true>)
                           : (p.no_delta ? gdn_tc_bwd_kernel<true, false> : gdn_tc_bwd_kernel<false, false>);
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kBwdSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  e = launch_overlapped(kern, (unsigned)(num_seqs(p) * p.H), BT, kBwdSmemBytes, s, mq, mk, mv, mdo, mdq,
                        mdk, mdv, bp);
  prof_after(s, kTcBwd);
  return e;
}

}  // namespace gdn
