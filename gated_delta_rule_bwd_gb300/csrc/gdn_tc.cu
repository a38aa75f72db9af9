// Tensor-core (tcgen05 / TMEM / TMA) kernels for the GDN mixer: bf16 inputs,
// dk = dv = 128, chunk C = 64, fp32 state and accumulation.
//
// One CTA (128 threads = the 128 TMEM lanes) owns one (batch, head) sequence
// and walks its chunks in order.  The state is held transposed, G = H^T
// (dv x dk, row c = value dimension), as fp32 in registers (thread c owns
// row c) with a bf16 copy in shared memory as the MMA operand.  Per chunk
// (Q, K, V tiles of 64 x 128 loaded by TMA with 128-byte swizzle; gamma =
// within-chunk cumulative log gate, e = exp(gamma), f = exp(gamma_last -
// gamma), eC = exp(gamma_last)):
//
//   MMA1  [K;Q] K^T          -> K K^T (lanes 0-63), Q K^T (lanes 64-127)
//         A = strict_lower(beta_r K K^T o Gam),  P = lower(Q K^T o Gam)
//         T = (I + A)^-1 on CUDA cores (blocked 16 x 16 solve)
//         T' = T diag(beta e),  T'' = T diag(beta)
//   MMA2  W^T  = K^T T'^T                       (W = T diag(beta e) K)
//   MMA3  U^T  = V^T T''^T - G W^T              (U = T diag(beta)(V - eK H))
//   MMA4  O^T  = G (eQ)^T + U^T P^T             (O = diag(e) Q H + P U)
//   MMA5  dG   = (U diag(f))^T K                (G' = eC G + dG)
//
// Every product has M = 128.  The TMA tiles of K and V serve both as K-major
// operands (rows = tokens) and, through MN-major descriptors, as their own
// transposes, so nothing is transposed in software.  MMAs are issued by one
// thread and complete on an mbarrier; every wait is bounded and a timeout is
// reported through the device status word instead of hanging.

#include <cuda.h>
#include <cudaTypedefs.h>

#include "gdn.h"
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {

// Per-device status word: bounded device-side waits record a timeout here.
__device__ int g_device_status = 0;

cudaError_t read_and_clear_device_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
  if (e != cudaSuccess) return e;
  *status = v;
  return cudaSuccess;
}

namespace {

using namespace tc;

constexpr int C = 64;     // chunk
constexpr int D = 128;    // dk = dv

// ---------------------------------------------------------------- shared memory map
// Offsets in bytes from a 1024-aligned base.  Stage s (double buffer) holds
// [K d0-63 | Q d0-63 | K d64-127 | Q d64-127] (8 KB each) then [V d0-63 | V d64-127].
constexpr int kStageKQ = 0;
constexpr int kStageV = 32768;
constexpr int kStageBytes = 49152;
constexpr int kOffStage0 = 0;
constexpr int kOffG = 2 * kStageBytes;          // G bf16, K-major [c][d], 2 x 16 KB
constexpr int kOffT1 = kOffG + 32768;           // T' [r][j] K-major          (8 KB)
constexpr int kOffT2 = kOffT1 + 8192;           // T'' [r][j]                  (8 KB)
constexpr int kOffP = kOffT2 + 8192;            // P [r][j]                    (8 KB)
constexpr int kOffW = kOffP + 8192;             // W, MN-major rows d, 64 r   (16 KB)
constexpr int kOffU = kOffW + 16384;            // U^T [c][j] K-major          (16 KB)
constexpr int kOffUf = kOffU + 16384;           // (U diag f)^T [c][j]         (16 KB)
// The fp32 solve scratch (A, T [64][65] and S [3][16][16]) aliases W / U / Uf:
// those are written only after the solve and its T', T'' outputs are done.
constexpr int kOffSolve = kOffW;
constexpr int kSolveBytes = (2 * 64 * 68 + 3 * 256) * 4;   // A, T [64][68] fp32 + S
static_assert(kSolveBytes <= 3 * 16384, "solve scratch must fit in W/U/Uf");
constexpr int kOffGate = kOffUf + 16384;         // gam, e, f, beta [64] each, eC
constexpr int kOffBar = kOffGate + 4 * 64 * 4 + 64;
constexpr int kSmemBytes = kOffBar + 128 + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

// TMEM columns
constexpr uint32_t kTmKQ = 0, kTmW = 64, kTmU = 128, kTmO = 192, kTmG = 256, kTmCols = 512;

struct FwdParams {
  const float* g;
  const float* beta;
  const float* h0;
  __nv_bfloat16* o;
  float* ht;
  __nv_bfloat16* states;  // optional: bf16 G tile of every chunk's entry state
                          // ([B*H][N][32 KB], shared-memory layout)
  const float* dht;       // with states: d(final state), for dht_dot
  float* dht_dot;         // with states: <dht, ht> per sequence
  int B, T, H, N;
};

// byte offset of element (row, col) in a K-major SW128 tile whose rows are
// 128 B (64 bf16) wide
__device__ __forceinline__ int sw_row_off(int row, int chunk16) {
  return row * 128 + ((chunk16 ^ (row & 7)) << 4);
}

__device__ __forceinline__ void cta_sync() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void report_timeout() { atomicExch(&g_device_status, GDN_ERR_DEVICE_TIMEOUT); }

// ---------------------------------------------------------------- forward kernel
//
// 512 threads: warp w reads TMEM lane quadrant q = w % 4 (lanes 32q..32q+31)
// and handles column group cg = w / 4 of every tile, so each epilogue is split
// four ways and every scheduler has four warps.  Thread (row, cg) owns
// columns [32 cg, 32 cg + 32) of state row `row`.

constexpr int FT = 512;              // forward threads
constexpr int kLdF = 68;             // fp32 row stride of the solve scratch (16-byte rows)

// 64-element row chunk helpers: write n16 groups of 8 bf16 (16 B) of a
// swizzled 128-byte row, starting at 16-byte chunk c0.
__device__ __forceinline__ void store_chunks(unsigned char* tile, int row, int c0, const float* v,
                                             int nchunks) {
  for (int k = 0; k < nchunks; ++k) {
    uint4 pk;
    uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(v[k * 8 + 2 * i], v[k * 8 + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(tile + sw_row_off(row, c0 + k)) = pk;
  }
}

// T = (I + A)^-1 for a 64 x 64 strictly lower A (fp32, row stride kLdF), by
// 16 x 16 blocks; all FT threads take part.
__device__ void solve_unit_lower_f(const float* A, float* T, float* S) {
  const int tid = threadIdx.x;
  if (tid < 64) {
    const int ib = tid / 16, jj = tid % 16, o = ib * 16;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float s = (r == jj) ? 1.f : 0.f;
      if (r > jj) {
#pragma unroll
        for (int i = 0; i < r; ++i)
          if (i >= jj) s -= A[(o + r) * kLdF + o + i] * x[i];
      }
      x[r] = (r >= jj) ? s : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) T[(o + r) * kLdF + o + jj] = x[r];
  } else {
    // zero the strictly upper blocks (never read as T, but keep T well defined)
    for (int i = tid - 64; i < 64 * 64; i += FT - 64) {
      const int r = i / 64, c = i % 64;
      if ((c / 16) > (r / 16)) T[r * kLdF + c] = 0.f;
    }
  }
  __syncthreads();
  for (int L = 1; L < 4; ++L) {
    const int nb = 4 - L;
    for (int i = tid; i < nb * 256; i += FT) {
      const int b = i / 256, r = (i / 16) % 16, c = i % 16;
      const int ib = b + L, jb = b;
      float s = 0.f;
      for (int k = jb * 16; k < ib * 16; ++k) s += A[(ib * 16 + r) * kLdF + k] * T[k * kLdF + jb * 16 + c];
      S[b * 256 + r * 16 + c] = s;
    }
    __syncthreads();
    for (int i = tid; i < nb * 256; i += FT) {
      const int b = i / 256, r = (i / 16) % 16, c = i % 16;
      const int ib = b + L, jb = b;
      float s = 0.f;
      for (int k = 0; k <= r; ++k) s += T[(ib * 16 + r) * kLdF + ib * 16 + k] * S[b * 256 + k * 16 + c];
      T[(ib * 16 + r) * kLdF + jb * 16 + c] = -s;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(FT, 1)
gdn_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, cg = warp >> 2;
  const int row = quad * 32 + lane;    // TMEM lane / tile row owned by this thread
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;

  float* gam = reinterpret_cast<float*>(sm + kOffGate);
  float* ee = gam + 64;
  float* ff = ee + 64;
  float* bt = ff + 64;
  float* eC = bt + 64;
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + kOffBar);  // [2]
  uint64_t* bar_mma = bar_load + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  float* Am = reinterpret_cast<float*>(sm + kOffSolve);
  float* Tm = Am + 64 * kLdF;
  float* Sm = Tm + 64 * kLdF;

  if (tid == 0) {
    mbar_init(&bar_load[0], 1);
    mbar_init(&bar_load[1], 1);
    mbar_init(bar_mma, 1);
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

  auto issue_load = [&](int ci) {
    unsigned char* st = sm + kOffStage0 + (ci & 1) * kStageBytes;
    uint64_t* bar = &bar_load[ci & 1];
    mbar_arrive_expect_tx(bar, 6 * 8192);
    const int t0 = ci * C;
    tma_load_4d(st + kStageKQ + 0, &tm_k, bar, 0, h, t0, b);
    tma_load_4d(st + kStageKQ + 8192, &tm_q, bar, 0, h, t0, b);
    tma_load_4d(st + kStageKQ + 16384, &tm_k, bar, 64, h, t0, b);
    tma_load_4d(st + kStageKQ + 24576, &tm_q, bar, 64, h, t0, b);
    tma_load_4d(st + kStageV + 0, &tm_v, bar, 0, h, t0, b);
    tma_load_4d(st + kStageV + 8192, &tm_v, bar, 64, h, t0, b);
  };
  auto state_dst = [&](int ci) -> unsigned char* {
    return p.states ? reinterpret_cast<unsigned char*>(p.states) +
                          ((size_t)bh * p.N + ci) * (size_t)(2 * 16384)
                    : nullptr;
  };
  const bool want_o = p.o != nullptr;
  // this thread's 32 state columns: d in [32 cg, 32 cg + 32) = tile region cg/2, chunks 4(cg%2)..
  const int g_region = cg >> 1, g_chunk0 = (cg & 1) * 4;
  auto write_g = [&](const float* Gv, unsigned char* dst) {
    unsigned char* tile = sm + kOffG + g_region * 16384;
    for (int k = 0; k < 4; ++k) {
      uint4 pk;
      uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(Gv[k * 8 + 2 * i], Gv[k * 8 + 2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      const int off = sw_row_off(row, g_chunk0 + k);
      *reinterpret_cast<uint4*>(tile + off) = pk;
      if (dst) *reinterpret_cast<uint4*>(dst + g_region * 16384 + off) = pk;
    }
  };

  float G[32];
#pragma unroll
  for (int i = 0; i < 32; ++i)
    G[i] = p.h0 ? p.h0[((size_t)bh * D + cg * 32 + i) * D + row] : 0.f;
  write_g(G, state_dst(0));

  // gate prefetch (warp 0): registers for the next chunk
  float pg0 = 0.f, pg1 = 0.f, pb0 = 0.f, pb1 = 0.f;
  auto load_gates = [&](int ci) {
    const int t0 = ci * C, n = min(C, p.T - t0);
    const size_t base = ((size_t)b * p.T + t0) * p.H + h;
    pg0 = lane < n ? p.g[base + (size_t)lane * p.H] : 0.f;
    pg1 = lane + 32 < n ? p.g[base + (size_t)(lane + 32) * p.H] : 0.f;
    pb0 = lane < n ? p.beta[base + (size_t)lane * p.H] : 0.f;
    pb1 = lane + 32 < n ? p.beta[base + (size_t)(lane + 32) * p.H] : 0.f;
  };
  if (warp == 0) load_gates(0);
  fence_async_shared();
  if (tid == 0) issue_load(0);
  cta_sync();

  uint32_t mma_phase = 0;
  uint32_t load_phase[2] = {0, 0};
  bool ok = true;
  auto mma_wait = [&]() {
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
  };

  for (int ci = 0; ci < p.N && ok; ++ci) {
    const int s = ci & 1, t0 = ci * C, n = min(C, p.T - t0);
    unsigned char* st = sm + kOffStage0 + s * kStageBytes;
    const uint32_t st_kq = smem_u32(st + kStageKQ), st_v = smem_u32(st + kStageV);

    if (warp == 0) {
      float g0 = pg0, g1 = pg1;
      bt[lane] = pb0;
      bt[lane + 32] = pb1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        float a0 = __shfl_up_sync(0xffffffffu, g0, off);
        float a1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (lane >= off) g0 += a0, g1 += a1;
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float gl = __shfl_sync(0xffffffffu, g1, 31);
      gam[lane] = g0;
      gam[lane + 32] = g1;
      ee[lane] = __expf(g0);
      ee[lane + 32] = __expf(g1);
      ff[lane] = __expf(gl - g0);
      ff[lane + 32] = __expf(gl - g1);
      if (lane == 0) *eC = __expf(gl);
      if (ci + 1 < p.N) load_gates(ci + 1);
    }
    ok = __syncthreads_and(mbar_wait(&bar_load[s], load_phase[s]));
    load_phase[s] ^= 1;
    if (!ok) break;
    if (tid == 0) {
      // MMA1: [K;Q] K^T, M=128 N=64 K=128
      const uint32_t idesc = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        mma_bf16(tmem + kTmKQ, sw128_desc(st_kq + off, 16, 1024), sw128_desc(st_kq + off, 16, 1024),
                 idesc, ks > 0);
      }
      mma_commit(bar_mma);
      if (ci + 1 < p.N) issue_load(ci + 1);
    }
    mma_wait();
    if (!ok) break;

    // E1: rows 0-63: A (fp32); rows 64-127: P (bf16); this thread: 16 columns
    {
      float v[16];
      tmem_ld16(tmem + lane_base + kTmKQ + cg * 16, v);
      if (row < 64) {
        const int r = row;
        const float gr = gam[r], br = bt[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          v[i] = (j < r) ? br * v[i] * __expf(gr - gam[j]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(Am + r * kLdF + cg * 16 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else {
        const int r = row - 64;
        const float gr = gam[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          v[i] = (j <= r) ? v[i] * __expf(gr - gam[j]) : 0.f;
        }
        store_chunks(sm + kOffP, r, cg * 2, v, 2);
      }
    }
    cta_sync();
    solve_unit_lower_f(Am, Tm, Sm);
    // T' = T diag(beta e), T'' = T diag(beta): one 16-byte chunk per thread
    {
      const int r = tid >> 3, c8 = tid & 7;
      float v1[8], v2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = c8 * 8 + i;
        const float t = (j <= r) ? Tm[r * kLdF + j] : 0.f;
        v2[i] = t * bt[j];
        v1[i] = v2[i] * ee[j];
      }
      store_chunks(sm + kOffT1, r, c8, v1, 1);
      store_chunks(sm + kOffT2, r, c8, v2, 1);
    }
    // scale Q rows in place by e_r (Q is done as an MMA1 operand): 2 chunks per thread
    for (int i = tid; i < 2 * 64 * 8; i += FT) {
      const int half = i / 512, r = (i / 8) % 64, c8 = i % 8;
      uint4* ptr = reinterpret_cast<uint4*>(st + kStageKQ + half * 16384 + 8192 + r * 128 + c8 * 16);
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
    if (tid == 0) {
      // MMA2: W^T = K^T T'^T  (A: K tile MN-major, M=d; B: T' K-major, N=r)
      const uint32_t id2 = idesc_bf16(128, 64, true, false);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kTmW, sw128_desc(st_kq + ks * 2048, 16384, 1024),
                 sw128_desc(smem_u32(sm + kOffT1) + ks * 32, 16, 1024), id2, ks > 0);
      // MMA3a: U^T = V^T T''^T  (A: V tile MN-major, M=c)
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kTmU, sw128_desc(st_v + ks * 2048, 8192, 1024),
                 sw128_desc(smem_u32(sm + kOffT2) + ks * 32, 16, 1024), id2, ks > 0);
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // E2: W^T row d -> W tile (MN-major: row d holds 64 r)
    {
      float w[16];
      tmem_ld16(tmem + lane_base + kTmW + cg * 16, w);
      store_chunks(sm + kOffW, row, cg * 2, w, 2);
    }
    fence_async_shared();
    cta_sync();
    if (tid == 0) {
      // MMA3b: U^T += -G W^T (A: G K-major M=c K=d; B: W MN-major N=r K=d)
      const uint32_t id3 = idesc_bf16(128, 64, false, true, true);
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kTmU, sw128_desc(smem_u32(sm + kOffG) + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024),
                 sw128_desc(smem_u32(sm + kOffW) + ks * 2048, 16384, 1024), id3, 1);
      // MMA4a: O^T = G (eQ)^T (B: Q tile K-major N=r K=d)
      const uint32_t id4 = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < (want_o ? 8 : 0); ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        mma_bf16(tmem + kTmO, sw128_desc(smem_u32(sm + kOffG) + off, 16, 1024),
                 sw128_desc(st_kq + 8192 + off, 16, 1024), id4, ks > 0);
      }
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // E3: U^T row c -> U^T tile and (U diag f)^T tile
    {
      float u[16];
      tmem_ld16(tmem + lane_base + kTmU + cg * 16, u);
      store_chunks(sm + kOffU, row, cg * 2, u, 2);
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] *= ff[cg * 16 + i];
      store_chunks(sm + kOffUf, row, cg * 2, u, 2);
    }
    fence_async_shared();
    cta_sync();
    if (tid == 0) {
      // MMA4b: O^T += U^T P^T (A: U^T K-major M=c K=j; B: P K-major N=r K=j)
      const uint32_t id4 = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < (want_o ? 4 : 0); ++ks)
        mma_bf16(tmem + kTmO, sw128_desc(smem_u32(sm + kOffU) + ks * 32, 16, 1024),
                 sw128_desc(smem_u32(sm + kOffP) + ks * 32, 16, 1024), id4, 1);
      // MMA5: dG = (U diag f)^T K (B: K tile MN-major, N=d (2 atoms), K=j)
      const uint32_t id5 = idesc_bf16(128, 128, false, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kTmG, sw128_desc(smem_u32(sm + kOffUf) + ks * 32, 16, 1024),
                 sw128_desc(st_kq + ks * 2048, 16384, 1024), id5, ks > 0);
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // E4: O^T row c, columns r in [16 cg, 16 cg + 16) -> o[b, t0 + r, h, c]
    if (want_o) {
      float v[16];
      tmem_ld16(tmem + lane_base + kTmO + cg * 16, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = cg * 16 + i;
        if (r < n) p.o[(((size_t)b * p.T + t0 + r) * p.H + h) * D + row] = __float2bfloat16_rn(v[i]);
      }
    }
    // E5: G = eC G + dG on this thread's 32 columns; bf16 copy for the next chunk
    {
      const float ec = *eC;
      float v32[32];
      tmem_ld32(tmem + lane_base + kTmG + cg * 32, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) G[i] = fmaf(ec, G[i], v32[i]);
      write_g(G, ci + 1 < p.N ? state_dst(ci + 1) : nullptr);
    }
    fence_async_shared();
    cta_sync();
  }

  if (!ok) {
    if (tid == 0) report_timeout();
    // let any tile load still in flight land before the CTA exits (bounded)
    for (int s2 = 0; s2 < 2; ++s2) mbar_wait(&bar_load[s2], load_phase[s2], 1u << 20);
  } else {
    if (p.ht) {
#pragma unroll
      for (int i = 0; i < 32; ++i) p.ht[((size_t)bh * D + cg * 32 + i) * D + row] = G[i];
    }
    if (p.dht_dot) {
      float acc = 0.f;
      if (p.dht) {
#pragma unroll
        for (int i = 0; i < 32; ++i) acc += p.dht[((size_t)bh * D + cg * 32 + i) * D + row] * G[i];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      float* red = reinterpret_cast<float*>(sm + kOffGate);  // gates are no longer needed
      __syncthreads();
      if (lane == 0) red[warp] = acc;
      __syncthreads();
      if (tid == 0) {
        float t = 0.f;
        for (int w = 0; w < FT / 32; ++w) t += red[w];
        p.dht_dot[bh] = t;
      }
    }
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

// ---------------------------------------------------------------- backward kernel
//
// Reverse chunk scan, one CTA per sequence.  The running state gradient is
// held transposed, dG = dH^T (dv x dk), fp32 in registers (thread c owns row
// c) with a bf16 copy in shared memory.  Each chunk's entry state G_in comes
// from the workspace (written by the forward kernel in states mode).  With
// R = V - diag(e) K H_in, U = T diag(beta) R, T = (I + A)^-1:
//
//   MMA1  [K;Q] K^T                -> K K^T (kept in TMEM), Q K^T -> P
//   MMA   -G_in K^T                -> R^T = V^T + (-G_in K^T) diag(e)
//   MMA   dG K^T, dO^T P           -> dU^T = (dG K^T) diag(f) + dO^T P
//   MMA   U^T = (R^T diag beta) T^T,  dZ^T = dU^T T     (dZ = (I+A)^-T dU)
//   MMA   [dZ; dO] U^T             -> dA = -strict_lower(dZ U^T), dP = dO U^T
//   MMA   dG_in = eC dG + (e dO)^T Q - (e dR)^T K       (dR = diag(beta) dZ)
//   MMA   dQ^T = G_in^T (e dO)^T + K^T (dP o Gam)^T
//   MMA   dK^T = dG^T (U diag f)^T - G_in^T (e dR)^T... + Q^T (dP o Gam)
//               + K^T (M + M^T),  M = diag(beta) dA o Gam
//
// dv = dR; dbeta_r = sum_c dZ_rc R_rc + sum_j dA_rj (K K^T o Gam)_rj.  The
// log-gate gradient uses the scaling identity of the scalar gate inside each
// chunk: dg_t = sum_{s >= t in the chunk} (q_s . dq_s - v_s . dv_s) +
// <dH_out, H_out>, where <dH_out, H_out> is <dH_in, H_in> of the next chunk
// (or <dht, ht> for the last one).  Keeping the sum inside the chunk avoids
// accumulating the rounding of thousands of terms.

constexpr int BT = 512;                  // backward threads (as the forward)
constexpr int kB_KQ = 0;                 // [Kh0 | Qh0 | Kh1 | Qh1]
constexpr int kB_ZO = 32768;             // [dZh0 | dOh0 | dZh1 | dOh1]
constexpr int kB_GI = 65536;             // G_in tile (K-major [c][d])
constexpr int kB_DG = 98304;             // dG tile (K-major [c][d])
constexpr int kB_V = 131072;             // [Vh0 | Vh1]
constexpr int kB_T = kB_V + 16384;       // T [r][j]; after the dZ product: M = beta dA o Gam
constexpr int kB_P = kB_T + 8192;        // P [r][j]; after dO^T P: dP o Gam
constexpr int kB_X = kB_P + 8192;        // three 16 KB slots, reused by phase
constexpr int kB_GATE = kB_X + 3 * 16384;  // gam, e, f, beta, db1, db2, dlc [64] each
constexpr int kB_RED = kB_GATE + 7 * 256;  // reduction scratch [16][64] floats
constexpr int kB_EC = kB_RED + 4096;
constexpr int kB_BAR = kB_EC + 64;
constexpr int kBwdSmemBytes = kB_BAR + 128 + 1024;
static_assert(kSolveBytes <= 3 * 16384, "solve scratch fits the X slots");
static_assert(kBwdSmemBytes <= 227 * 1024, "shared memory budget");

// TMEM columns of the backward kernel
constexpr uint32_t kBtKQ = 0, kBtR = 64, kBtX1 = 128, kBtX2 = 192, kBtU = 256, kBtZ = 320,
                   kBtG3 = 384;  // G3: 128 columns
// reused later: G4 -> X1 columns, dQ -> X2 columns, dK -> U columns

struct BwdParams {
  const float* g;
  const float* beta;
  const float* dht;
  const float* dht_dot;          // <dht, ht> per sequence (workspace)
  const unsigned char* states;   // [B*H][N][32 KB]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  float* dg;
  float* dbeta;
  float* dh0;
  int B, T, H, N;
};

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Each thread holds v[i] for tile column (16 cg + i) of its row; returns in
// out[r] (r < 64) the sum over all 128 rows.  Within a warp: four halving
// exchanges and one pairwise add (lane l ends with column 16 cg + l/2); across
// the four warps of a column group: red[16][16] in shared memory.
__device__ __forceinline__ void cta_sum_rows16(float (&v)[16], float* red, float* out) {
  const int l = threadIdx.x & 31, w = threadIdx.x >> 5, quad = w & 3, cg = w >> 2;
#pragma unroll
  for (int step = 0; step < 4; ++step) {
    const int off = 16 >> step, half = 8 >> step;
    const bool up = (l & off) != 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (i < half) {
        const float send = up ? v[i] : v[i + half];
        const float keep = up ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
  }
  v[0] += __shfl_xor_sync(0xffffffffu, v[0], 1);
  if ((l & 1) == 0) red[(cg * 4 + quad) * 16 + (l >> 1)] = v[0];
  __syncthreads();
  if (threadIdx.x < 64) {
    const int c = threadIdx.x >> 4, i = threadIdx.x & 15;
    out[threadIdx.x] = red[(c * 4 + 0) * 16 + i] + red[(c * 4 + 1) * 16 + i] +
                       red[(c * 4 + 2) * 16 + i] + red[(c * 4 + 3) * 16 + i];
  }
  __syncthreads();
}

// bf16 element (row, col) of a swizzled 64-wide K-major tile
__device__ __forceinline__ float tile_elem(const unsigned char* tile, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
      tile + sw_row_off(row, col >> 3) + (col & 7) * 2));
}

__global__ void __launch_bounds__(BT, 1)
gdn_tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  BwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32, lane = tid & 31;
  const int quad = warp & 3, cg = warp >> 2;
  const int row = quad * 32 + lane;
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;

  float* gam = reinterpret_cast<float*>(sm + kB_GATE);
  float* ee = gam + 64;
  float* ff = ee + 64;
  float* bt = ff + 64;
  float* db1 = bt + 64;
  float* db2 = db1 + 64;
  float* dlc = db2 + 64;
  float* red = reinterpret_cast<float*>(sm + kB_RED);
  float* eC = reinterpret_cast<float*>(sm + kB_EC);
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + kB_BAR);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  float* Am = reinterpret_cast<float*>(sm + kB_X);
  float* Tm = Am + 64 * kLdF;
  float* Sm = Tm + 64 * kLdF;
  const uint32_t sKQ = smem_u32(sm + kB_KQ), sZO = smem_u32(sm + kB_ZO);
  const uint32_t sGI = smem_u32(sm + kB_GI), sDG = smem_u32(sm + kB_DG);
  const uint32_t sT = smem_u32(sm + kB_T), sP = smem_u32(sm + kB_P);
  const uint32_t sDP = sP, sM = sT;
  const uint32_t sX0 = smem_u32(sm + kB_X), sX1 = sX0 + 16384, sX2 = sX0 + 32768;

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
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

  // this thread's 32 state-gradient columns: d in [32 cg, 32 cg + 32)
  const int g_region = cg >> 1, g_chunk0 = (cg & 1) * 4;
  float dG[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) dG[i] = p.dht ? p.dht[((size_t)bh * D + cg * 32 + i) * D + row] : 0.f;
  auto write_dg = [&]() {
    unsigned char* tile = sm + kB_DG + g_region * 16384;
    for (int k = 0; k < 4; ++k) {
      uint4 pk;
      uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(dG[k * 8 + 2 * i], dG[k * 8 + 2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      *reinterpret_cast<uint4*>(tile + sw_row_off(row, g_chunk0 + k)) = pk;
    }
  };
  write_dg();
  // <dH_out, H_out> of the chunk being processed (the last chunk: <dht, ht>)
  float carry = p.dht_dot ? p.dht_dot[bh] : 0.f;

  float pg0 = 0.f, pg1 = 0.f, pb0 = 0.f, pb1 = 0.f;
  auto load_gates = [&](int ci) {
    const int t0 = ci * C, n = min(C, p.T - t0);
    const size_t base = ((size_t)b * p.T + t0) * p.H + h;
    pg0 = lane < n ? p.g[base + (size_t)lane * p.H] : 0.f;
    pg1 = lane + 32 < n ? p.g[base + (size_t)(lane + 32) * p.H] : 0.f;
    pb0 = lane < n ? p.beta[base + (size_t)lane * p.H] : 0.f;
    pb1 = lane + 32 < n ? p.beta[base + (size_t)(lane + 32) * p.H] : 0.f;
  };
  if (warp == 0) load_gates(p.N - 1);

  uint32_t mma_phase = 0, load_phase = 0;
  bool ok = true;
  auto mma_wait = [&]() {
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
  };

  for (int ci = p.N - 1; ci >= 0 && ok; --ci) {
    const int t0 = ci * C, n = min(C, p.T - t0);
    fence_async_shared();
    cta_sync();
    if (tid == 0) {
      mbar_arrive_expect_tx(bar_load, 8 * 8192 + 32768);
      tma_load_4d(sm + kB_KQ + 0, &tm_k, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_KQ + 8192, &tm_q, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_KQ + 16384, &tm_k, bar_load, 64, h, t0, b);
      tma_load_4d(sm + kB_KQ + 24576, &tm_q, bar_load, 64, h, t0, b);
      tma_load_4d(sm + kB_ZO + 8192, &tm_do, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_ZO + 24576, &tm_do, bar_load, 64, h, t0, b);
      tma_load_4d(sm + kB_V, &tm_v, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_V + 8192, &tm_v, bar_load, 64, h, t0, b);
      bulk_load(sm + kB_GI, p.states + ((size_t)bh * p.N + ci) * 32768, 32768, bar_load);
    }
    if (warp == 0) {
      float g0 = pg0, g1 = pg1;
      bt[lane] = pb0;
      bt[lane + 32] = pb1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        float a0 = __shfl_up_sync(0xffffffffu, g0, off);
        float a1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (lane >= off) g0 += a0, g1 += a1;
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float gl = __shfl_sync(0xffffffffu, g1, 31);
      gam[lane] = g0;
      gam[lane + 32] = g1;
      ee[lane] = __expf(g0);
      ee[lane + 32] = __expf(g1);
      ff[lane] = __expf(gl - g0);
      ff[lane + 32] = __expf(gl - g1);
      if (lane == 0) *eC = __expf(gl);
      if (ci > 0) load_gates(ci - 1);
    }
    ok = __syncthreads_and(mbar_wait(bar_load, load_phase));
    load_phase ^= 1;
    if (!ok) break;
    // ---- MMA1: [K;Q] K^T
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        mma_bf16(tmem + kBtKQ, sw128_desc(sKQ + off, 16, 1024), sw128_desc(sKQ + off, 16, 1024), id,
                 ks > 0);
      }
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    {
      float v[16];
      tmem_ld16(tmem + lb + kBtKQ + cg * 16, v);
      if (row < 64) {
        const int r = row;
        const float gr = gam[r], br = bt[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          v[i] = (j < r) ? br * v[i] * __expf(gr - gam[j]) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; i += 4)
          *reinterpret_cast<float4*>(Am + r * kLdF + cg * 16 + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
      } else {
        const int r = row - 64;
        const float gr = gam[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          v[i] = (j <= r) ? v[i] * __expf(gr - gam[j]) : 0.f;
        }
        store_chunks(sm + kB_P, r, cg * 2, v, 2);
      }
    }
    cta_sync();
    solve_unit_lower_f(Am, Tm, Sm);
    {
      const int r = tid >> 3, c8 = tid & 7;
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = c8 * 8 + i;
        v[i] = (j <= r) ? Tm[r * kLdF + j] : 0.f;
      }
      store_chunks(sm + kB_T, r, c8, v, 1);
    }
    fence_async_shared();
    cta_sync();
    // ---- -G_in K^T, dG K^T, dO^T P
    if (tid == 0) {
      const uint32_t idn = idesc_bf16(128, 64, false, false, true);
      const uint32_t id = idesc_bf16(128, 64, false, false);
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t off = (ks / 4) * 16384 + (ks % 4) * 32;
        mma_bf16(tmem + kBtR, sw128_desc(sGI + off, 16, 1024), sw128_desc(sKQ + off, 16, 1024), idn,
                 ks > 0);
        mma_bf16(tmem + kBtX1, sw128_desc(sDG + off, 16, 1024), sw128_desc(sKQ + off, 16, 1024), id,
                 ks > 0);
      }
      const uint32_t idmm = idesc_bf16(128, 64, true, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtX2, sw128_desc(sZO + 8192 + ks * 2048, 16384, 1024),
                 sw128_desc(sP + ks * 2048, 16384, 1024), idmm, ks > 0);
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // ---- E3: beta R^T -> X0, dU^T -> X1  (this thread: row c, columns 16 cg + i)
    {
      float a[16], x[16];
      tmem_ld16(tmem + lb + kBtR + cg * 16, a);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = cg * 16 + i;
        a[i] = bt[r] * (tile_elem(sm + kB_V + (row >> 6) * 8192, r, row & 63) + ee[r] * a[i]);
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
    // ---- E4: U^T -> X0, (U diag f)^T -> X2, e dR^T -> X1, dZ rows -> ZO, dv, dbeta part 1
    float acc[16];  // this thread's terms of the log-gate gradient, columns 16 cg + i
    {
      float u[16];
      tmem_ld16(tmem + lb + kBtU + cg * 16, u);
      store_chunks(sm + kB_X, row, cg * 2, u, 2);
#pragma unroll
      for (int i = 0; i < 16; ++i) u[i] *= ff[cg * 16 + i];
      store_chunks(sm + kB_X + 32768, row, cg * 2, u, 2);
      float z[16], rr[16];
      tmem_ld16(tmem + lb + kBtZ + cg * 16, z);
      tmem_ld16(tmem + lb + kBtR + cg * 16, rr);
      const int half = row >> 6, cc = row & 63;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = cg * 16 + i;
        const float vr = tile_elem(sm + kB_V + half * 8192, r, cc);
        const float dr = bt[r] * z[i];
        if (r < n) p.dv[(((size_t)b * p.T + t0 + r) * p.H + h) * D + row] = __float2bfloat16_rn(dr);
        acc[i] = -vr * dr;                        // -v . dv
        rr[i] = z[i] * (vr + ee[r] * rr[i]);      // dZ_rc R_rc
        *reinterpret_cast<__nv_bfloat16*>(sm + kB_ZO + half * 16384 + sw_row_off(r, cc >> 3) +
                                          (cc & 7) * 2) = __float2bfloat16_rn(z[i]);
        z[i] = ee[r] * dr;
      }
      store_chunks(sm + kB_X + 16384, row, cg * 2, z, 2);
      cta_sum_rows16(rr, red, db1);
    }
    fence_async_shared();
    cta_sync();
    // ---- G4: [dZ; dO] U^T  (lanes 0-63: dZ U^T, lanes 64-127: dO U^T)
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, 64, false, true);
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtX1, sw128_desc(sZO + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024),
                 sw128_desc(sX0 + ks * 2048, 16384, 1024), id, ks > 0);
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    {
      float x[16];
      tmem_ld16(tmem + lb + kBtX1 + cg * 16, x);
      if (row < 64) {
        // dA = -strict_lower(dZ U^T); dbeta part 2; M = beta dA o Gam
        const int r = row;
        float kk[16];
        tmem_ld16(tmem + lb + kBtKQ + cg * 16, kk);
        const float gr = gam[r], br = bt[r];
        float s2 = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          const float w = (j < r) ? __expf(gr - gam[j]) : 0.f;
          const float da = -x[i];
          s2 += da * kk[i] * w;
          x[i] = br * da * w;
        }
        red[cg * 64 + r] = s2;
        store_chunks(sm + kB_T, r, cg * 2, x, 2);
      } else {
        const int r = row - 64;
        const float gr = gam[r];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = cg * 16 + i;
          x[i] = (j <= r) ? x[i] * __expf(gr - gam[j]) : 0.f;
        }
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
    if (tid < 64) db2[tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
    // ---- dG_in part, dQ^T, dK^T
    if (tid == 0) {
      // G3 = (e dO)^T Q - (e dR)^T K   [c x d]
      const uint32_t idg = idesc_bf16(128, 128, true, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtG3, sw128_desc(sZO + 8192 + ks * 2048, 16384, 1024),
                 sw128_desc(sKQ + 8192 + ks * 2048, 16384, 1024), idg, ks > 0);
      const uint32_t idgn = idesc_bf16(128, 128, false, true, true);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtG3, sw128_desc(sX1 + ks * 32, 16, 1024), sw128_desc(sKQ + ks * 2048, 16384, 1024),
                 idgn, 1);
      // dQ^T = G_in^T (e dO)^T + K^T (dP o Gam)^T   [d x r]  -> X2 columns
      const uint32_t idq = idesc_bf16(128, 64, true, false);
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtX2, sw128_desc(sGI + ks * 2048, 16384, 1024),
                 sw128_desc(sZO + 8192 + (ks / 4) * 16384 + (ks % 4) * 32, 16, 1024), idq, ks > 0);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtX2, sw128_desc(sKQ + ks * 2048, 16384, 1024), sw128_desc(sDP + ks * 32, 16, 1024),
                 idq, 1);
      // dK^T  [d x j] -> U columns
      const uint32_t idmm = idesc_bf16(128, 64, true, true);
      const uint32_t idmmn = idesc_bf16(128, 64, true, true, true);
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtU, sw128_desc(sDG + ks * 2048, 16384, 1024), sw128_desc(sX2 + ks * 2048, 16384, 1024),
                 idmm, ks > 0);
      for (int ks = 0; ks < 8; ++ks)
        mma_bf16(tmem + kBtU, sw128_desc(sGI + ks * 2048, 16384, 1024), sw128_desc(sX1 + ks * 2048, 16384, 1024),
                 idmmn, 1);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtU, sw128_desc(sKQ + 8192 + ks * 2048, 16384, 1024),
                 sw128_desc(sDP + ks * 2048, 16384, 1024), idmm, 1);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtU, sw128_desc(sKQ + ks * 2048, 16384, 1024), sw128_desc(sM + ks * 32, 16, 1024),
                 idq, 1);
      for (int ks = 0; ks < 4; ++ks)
        mma_bf16(tmem + kBtU, sw128_desc(sKQ + ks * 2048, 16384, 1024), sw128_desc(sM + ks * 2048, 16384, 1024),
                 idmm, 1);
      mma_commit(bar_mma);
    }
    mma_wait();
    if (!ok) break;
    // ---- E6: dG update, dq (+ q.dq), dk, dbeta, dg
    {
      const float ec = *eC;
      float v32[32];
      tmem_ld32(tmem + lb + kBtG3 + cg * 32, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) dG[i] = fmaf(ec, dG[i], v32[i]);
      float x[16];
      tmem_ld16(tmem + lb + kBtX2 + cg * 16, x);  // dQ^T row d = row, columns r = 16 cg + i
      const int half = row >> 6, cc = row & 63;
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = cg * 16 + i;
        acc[i] += tile_elem(sm + kB_KQ + half * 16384 + 8192, r, cc) * x[i];
        if (r < n) p.dq[(((size_t)b * p.T + t0 + r) * p.H + h) * D + row] = __float2bfloat16_rn(x[i]);
      }
      tmem_ld16(tmem + lb + kBtU + cg * 16, x);  // dK^T row d, columns j
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int j = cg * 16 + i;
        if (j < n) p.dk[(((size_t)b * p.T + t0 + j) * p.H + h) * D + row] = __float2bfloat16_rn(x[i]);
      }
    }
    cta_sum_rows16(acc, red, dlc);
    if (tid < 64) {
      const int r = tid;
      if (r < n) p.dbeta[((size_t)b * p.T + t0 + r) * p.H + h] = db1[r] + db2[r];
    }
    // <dH_in, H_in> of this chunk = <dH_out, H_out> of the chunk before it
    float dot = 0.f;
    {
      const unsigned char* tile = sm + kB_GI + g_region * 16384;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 pk = *reinterpret_cast<const uint4*>(tile + sw_row_off(row, g_chunk0 + k));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f2 = __bfloat1622float2(h2[i]);
          dot = fmaf(dG[k * 8 + 2 * i], f2.x, dot);
          dot = fmaf(dG[k * 8 + 2 * i + 1], f2.y, dot);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (lane == 0) red[256 + warp] = dot;
    __syncthreads();
    if (warp == 0) {
      // dg_t = sum_{s >= t, s in chunk} (q_s.dq_s - v_s.dv_s) + <dH_out, H_out>
      float a0 = dlc[lane], a1 = dlc[lane + 32];
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
      const size_t base = ((size_t)b * p.T + t0) * p.H + h;
      if (lane < n) p.dg[base + (size_t)lane * p.H] = carry + s0;
      if (lane + 32 < n) p.dg[base + (size_t)(lane + 32) * p.H] = carry + s1;
    }
    carry = 0.f;
#pragma unroll
    for (int w = 0; w < BT / 32; ++w) carry += red[256 + w];
    write_dg();
  }

  if (!ok) {
    if (tid == 0) report_timeout();
    mbar_wait(bar_load, load_phase, 1u << 20);
  } else if (p.dh0) {
#pragma unroll
    for (int i = 0; i < 32; ++i) p.dh0[((size_t)bh * D + cg * 32 + i) * D + row] = dG[i];
  }
  cta_sync();
  if (warp == 0) tmem_dealloc(tmem, kTmCols);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 4-D map over a [B, T, H, 128] bf16 tensor; box = 64 features x 1 head x
// 64 tokens x 1 batch row, 128-byte swizzle; rows past T read as zero.
cudaError_t make_token_map(CUtensorMap* m, const void* ptr, const Problem& p) {
  auto enc = get_encoder();
  if (!enc) return cudaErrorNotSupported;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.H, (cuuint64_t)p.T, (cuuint64_t)p.B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)p.H * D * 2, (cuuint64_t)p.T * p.H * D * 2};
  cuuint32_t box[4] = {64, 1, 64, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_fwd(const Problem& p, cudaStream_t s, bool want_out, __nv_bfloat16* states,
                       float* dht_dot) {
  CUtensorMap mq, mk, mv;
  cudaError_t e;
  if ((e = make_token_map(&mq, p.q, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mv, p.v, p)) != cudaSuccess) return e;
  FwdParams fp{p.g, p.beta, p.h0, want_out ? static_cast<__nv_bfloat16*>(p.o) : nullptr,
               want_out ? p.ht : nullptr, states, want_out ? nullptr : p.dht,
               dht_dot, p.B, p.T, p.H, p.N};
  e = cudaFuncSetAttribute(gdn_tc_fwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  gdn_tc_fwd_kernel<<<p.B * p.H, FT, kSmemBytes, s>>>(mq, mk, mv, fp);
  prof_after(s, want_out ? kTcFwd : kTcStates);
  return cudaGetLastError();
}

}  // namespace

bool tc_supported(const Problem& p) {
  return p.bf16 && !p.kda && p.dk == D && p.dv == D && p.C == C;
}

// Workspace of the tensor-core backward pass: the bf16 entry state of every
// chunk in MMA-operand layout (32 KB each), then <dht, ht> per sequence.
size_t tc_bwd_workspace(const Problem& p) {
  return align_up((size_t)p.B * p.H * p.N * 32768, 256) + align_up((size_t)p.B * p.H * 4, 256);
}

cudaError_t tc_fwd(const Problem& p, cudaStream_t s) {
  return launch_fwd(p, s, true, nullptr, nullptr);
}

cudaError_t tc_bwd(const Problem& p, cudaStream_t s) {
  unsigned char* ws = static_cast<unsigned char*>(p.ws);
  __nv_bfloat16* states = reinterpret_cast<__nv_bfloat16*>(ws);
  float* dht_dot = reinterpret_cast<float*>(ws + align_up((size_t)p.B * p.H * p.N * 32768, 256));
  cudaError_t e = launch_fwd(p, s, false, states, dht_dot);
  if (e != cudaSuccess) return e;
  CUtensorMap mq, mk, mv, mdo;
  if ((e = make_token_map(&mq, p.q, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mv, p.v, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdo, p.do_, p)) != cudaSuccess) return e;
  BwdParams bp{p.g, p.beta, p.dht, dht_dot,
               reinterpret_cast<const unsigned char*>(states), static_cast<__nv_bfloat16*>(p.dq),
               static_cast<__nv_bfloat16*>(p.dk_), static_cast<__nv_bfloat16*>(p.dv_), p.dg, p.dbeta,
               p.dh0, p.B, p.T, p.H, p.N};
  e = cudaFuncSetAttribute(gdn_tc_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kBwdSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  gdn_tc_bwd_kernel<<<p.B * p.H, BT, kBwdSmemBytes, s>>>(mq, mk, mv, mdo, bp);
  prof_after(s, kTcBwd);
  return cudaGetLastError();
}

}  // namespace gdn
