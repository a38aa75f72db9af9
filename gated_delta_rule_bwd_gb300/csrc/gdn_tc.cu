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
constexpr int NT = 128;   // threads per CTA

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
constexpr int kLdA = 65;
constexpr int kSolveBytes = (2 * 64 * kLdA + 3 * 256) * 4;
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

// Writes 64 fp32 values as one 128-byte swizzled bf16 row.
__device__ __forceinline__ void store_row64(unsigned char* tile, int row, const float* v) {
#pragma unroll
  for (int c8 = 0; c8 < 8; ++c8) {
    uint4 pk;
    uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(v[c8 * 8 + 2 * i], v[c8 * 8 + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(tile + sw_row_off(row, c8)) = pk;
  }
}

// Writes thread c's fp32 state row as row c of the bf16 G tile (two 64-wide
// column blocks of 16 KB) and, if dst is set, the same bytes to dst (a 32 KB
// global copy of the tile in its shared-memory layout).
__device__ __forceinline__ void store_g_tile(unsigned char* tile, const float* G, int row,
                                             unsigned char* dst) {
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
      uint4 pk;
      uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(G[half * 64 + c8 * 8 + 2 * i],
                                                  G[half * 64 + c8 * 8 + 2 * i + 1]);
        w[i] = *reinterpret_cast<uint32_t*>(&b2);
      }
      const int off = half * 16384 + sw_row_off(row, c8);
      *reinterpret_cast<uint4*>(tile + off) = pk;
      if (dst) *reinterpret_cast<uint4*>(dst + off) = pk;
    }
  }
}

__device__ __forceinline__ void cta_sync() {
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

__device__ __forceinline__ void report_timeout() { atomicExch(&g_device_status, GDN_ERR_DEVICE_TIMEOUT); }

// Unit-lower-triangular inverse T = (I + A)^-1 of a 64 x 64 strictly lower A
// (fp32, row stride kLdA), blocked in 16 x 16: diagonal blocks by forward
// substitution, off-diagonal blocks by T_ib,jb = -T_ib,ib sum_kb A_ib,kb T_kb,jb.
__device__ void solve_unit_lower(const float* A, float* T, float* S) {
  const int tid = threadIdx.x;
  for (int i = tid; i < 64 * 64; i += NT) T[(i / 64) * kLdA + (i % 64)] = 0.f;
  __syncthreads();
  if (tid < 64) {
    const int ib = tid / 16, jj = tid % 16, o = ib * 16;
    float x[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float s = (r == jj) ? 1.f : 0.f;
      if (r > jj) {
#pragma unroll
        for (int i = 0; i < r; ++i)
          if (i >= jj) s -= A[(o + r) * kLdA + o + i] * x[i];
      }
      x[r] = (r >= jj) ? s : 0.f;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) T[(o + r) * kLdA + o + jj] = x[r];
  }
  __syncthreads();
  for (int L = 1; L < 4; ++L) {
    const int nb = 4 - L;
    // S_b = sum_{kb=jb}^{ib-1} A[ib][kb] T[kb][jb],  block b: jb = b, ib = b + L
    for (int i = tid; i < nb * 256; i += NT) {
      const int b = i / 256, r = (i / 16) % 16, c = i % 16;
      const int ib = b + L, jb = b;
      float s = 0.f;
      for (int k = jb * 16; k < ib * 16; ++k) s += A[(ib * 16 + r) * kLdA + k] * T[k * kLdA + jb * 16 + c];
      S[b * 256 + r * 16 + c] = s;
    }
    __syncthreads();
    for (int i = tid; i < nb * 256; i += NT) {
      const int b = i / 256, r = (i / 16) % 16, c = i % 16;
      const int ib = b + L, jb = b;
      float s = 0.f;
      for (int k = 0; k <= r; ++k) s += T[(ib * 16 + r) * kLdA + ib * 16 + k] * S[b * 256 + k * 16 + c];
      T[(ib * 16 + r) * kLdA + jb * 16 + c] = -s;
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- forward kernel
__global__ void __launch_bounds__(NT, 1)
gdn_tc_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, FwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32;
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;

  float* gam = reinterpret_cast<float*>(sm + kOffGate);
  float* ee = gam + 64;
  float* ff = ee + 64;
  float* bt = ff + 64;
  float* eC = bt + 64;
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + kOffBar);  // [2]
  uint64_t* bar_mma = bar_load + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  float* Am = reinterpret_cast<float*>(sm + kOffSolve);
  float* Tm = Am + 64 * kLdA;
  float* Sm = Tm + 64 * kLdA;

  if (tid == 0) {
    mbar_init(&bar_load[0], 1);
    mbar_init(&bar_load[1], 1);
    mbar_init(bar_mma, 1);
    *abort_flag = 0;
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
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

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

  // state: thread c owns row c of G = H^T
  float G[D];
  {
#pragma unroll
    for (int d = 0; d < D; ++d)
      G[d] = p.h0 ? p.h0[((size_t)bh * D + d) * D + tid] : 0.f;
    store_g_tile(sm + kOffG, G, tid, state_dst(0));
  }
  fence_async_shared();
  if (tid == 0) issue_load(0);
  cta_sync();

  uint32_t mma_phase = 0;
  uint32_t load_phase[2] = {0, 0};
  bool ok = true;

  for (int ci = 0; ci < p.N && ok; ++ci) {
    const int s = ci & 1, t0 = ci * C, n = min(C, p.T - t0);
    unsigned char* st = sm + kOffStage0 + s * kStageBytes;
    const uint32_t st_kq = smem_u32(st + kStageKQ), st_v = smem_u32(st + kStageV);

    // gates of this chunk (warp 0): gamma = cumsum(g), e, f, eC
    if (warp == 0) {
      const int l = threadIdx.x;
      const size_t base = ((size_t)b * p.T + t0) * p.H + h;
      float g0 = l < n ? p.g[base + (size_t)l * p.H] : 0.f;
      float g1 = l + 32 < n ? p.g[base + (size_t)(l + 32) * p.H] : 0.f;
      bt[l] = l < n ? p.beta[base + (size_t)l * p.H] : 0.f;
      bt[l + 32] = l + 32 < n ? p.beta[base + (size_t)(l + 32) * p.H] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        float a0 = __shfl_up_sync(0xffffffffu, g0, off);
        float a1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (l >= off) g0 += a0, g1 += a1;
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float gl = __shfl_sync(0xffffffffu, g1, 31);
      gam[l] = g0;
      gam[l + 32] = g1;
      ee[l] = expf(g0);
      ee[l + 32] = expf(g1);
      ff[l] = expf(gl - g0);
      ff[l + 32] = expf(gl - g1);
      if (l == 0) *eC = expf(gl);
    }
    // tiles of this chunk
    ok = __syncthreads_and(mbar_wait(&bar_load[s], load_phase[s]));
    load_phase[s] ^= 1;
    if (tid == 0 && ok) {
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
    if (!ok) break;
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
    if (!ok) break;

    // E1: A (lanes 0-63) and P (lanes 64-127)
    {
      float kk[64];
      float v32[32];
      tmem_ld32(tmem + lane_base + kTmKQ, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) kk[i] = v32[i];
      tmem_ld32(tmem + lane_base + kTmKQ + 32, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) kk[32 + i] = v32[i];
      if (tid < 64) {
        const int r = tid;
        const float gr = gam[r], br = bt[r];
#pragma unroll
        for (int j = 0; j < 64; ++j) Am[r * kLdA + j] = (j < r) ? br * kk[j] * expf(gr - gam[j]) : 0.f;
      } else {
        const int r = tid - 64;
        const float gr = gam[r];
#pragma unroll
        for (int j = 0; j < 64; ++j) kk[j] = (j <= r) ? kk[j] * expf(gr - gam[j]) : 0.f;
        store_row64(sm + kOffP, r, kk);
      }
    }
    cta_sync();
    solve_unit_lower(Am, Tm, Sm);
    // T' = T diag(beta e), T'' = T diag(beta): thread -> (row r = tid/2, half)
    {
      const int r = tid >> 1, hf = tid & 1;
      float v1[32], v2[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int j = hf * 32 + i;
        const float t = (j <= r) ? Tm[r * kLdA + j] : 0.f;
        v2[i] = t * bt[j];
        v1[i] = v2[i] * ee[j];
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint4 p1, p2;
        uint32_t* w1 = reinterpret_cast<uint32_t*>(&p1);
        uint32_t* w2 = reinterpret_cast<uint32_t*>(&p2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __nv_bfloat162 a = __floats2bfloat162_rn(v1[c8 * 8 + 2 * i], v1[c8 * 8 + 2 * i + 1]);
          __nv_bfloat162 c2 = __floats2bfloat162_rn(v2[c8 * 8 + 2 * i], v2[c8 * 8 + 2 * i + 1]);
          w1[i] = *reinterpret_cast<uint32_t*>(&a);
          w2[i] = *reinterpret_cast<uint32_t*>(&c2);
        }
        *reinterpret_cast<uint4*>(sm + kOffT1 + sw_row_off(r, hf * 4 + c8)) = p1;
        *reinterpret_cast<uint4*>(sm + kOffT2 + sw_row_off(r, hf * 4 + c8)) = p2;
      }
    }
    // scale Q rows in place by e_r (Q is done as an MMA1 operand)
    for (int i = tid; i < 2 * 64 * 8; i += NT) {
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
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
    if (!ok) break;
    // E2: W^T row d -> W tile (MN-major: row d holds 64 r)
    {
      float w[64], v32[32];
      tmem_ld32(tmem + lane_base + kTmW, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) w[i] = v32[i];
      tmem_ld32(tmem + lane_base + kTmW + 32, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) w[32 + i] = v32[i];
      store_row64(sm + kOffW, tid, w);
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
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
    if (!ok) break;
    // E3: U^T row c -> U^T tile and (U diag f)^T tile
    {
      float u[64], v32[32];
      tmem_ld32(tmem + lane_base + kTmU, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) u[i] = v32[i];
      tmem_ld32(tmem + lane_base + kTmU + 32, v32);
#pragma unroll
      for (int i = 0; i < 32; ++i) u[32 + i] = v32[i];
      store_row64(sm + kOffU, tid, u);
#pragma unroll
      for (int j = 0; j < 64; ++j) u[j] *= ff[j];
      store_row64(sm + kOffUf, tid, u);
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
    ok = __syncthreads_and(mbar_wait(bar_mma, mma_phase));
    mma_phase ^= 1;
    tc_fence_after();
    if (!ok) break;
    // E4: O^T row c -> o[b, t0 + r, h, c]
    if (want_o) {
      float v32[32];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        tmem_ld32(tmem + lane_base + kTmO + half * 32, v32);
        {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int r = half * 32 + i;
            if (r < n) p.o[(((size_t)b * p.T + t0 + r) * p.H + h) * D + tid] = __float2bfloat16_rn(v32[i]);
          }
        }
      }
    }
    // E5: G = eC G + dG; bf16 copy for the next chunk
    {
      const float ec = *eC;
      float v32[32];
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tmem + lane_base + kTmG + q4 * 32, v32);
#pragma unroll
        for (int i = 0; i < 32; ++i) G[q4 * 32 + i] = fmaf(ec, G[q4 * 32 + i], v32[i]);
      }
      store_g_tile(sm + kOffG, G, tid, ci + 1 < p.N ? state_dst(ci + 1) : nullptr);
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
      for (int d = 0; d < D; ++d) p.ht[((size_t)bh * D + d) * D + tid] = G[d];
    }
    if (p.dht_dot) {
      // <dht, ht> over the sequence's whole state (row c = tid here)
      float acc = 0.f;
      if (p.dht) {
#pragma unroll
        for (int d = 0; d < D; ++d) acc += p.dht[((size_t)bh * D + d) * D + tid] * G[d];
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      float* red = reinterpret_cast<float*>(sm + kOffGate);  // gates are no longer needed
      __syncthreads();
      if ((tid & 31) == 0) red[warp] = acc;
      __syncthreads();
      if (tid == 0) p.dht_dot[bh] = red[0] + red[1] + red[2] + red[3];
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

constexpr int kB_KQ = 0;                 // [Kh0 | Qh0 | Kh1 | Qh1]
constexpr int kB_ZO = 32768;             // [dZh0 | dOh0 | dZh1 | dOh1]
constexpr int kB_GI = 65536;             // G_in tile (K-major [c][d])
constexpr int kB_DG = 98304;             // dG tile (K-major [c][d])
constexpr int kB_T = 131072;             // T [r][j]
constexpr int kB_P = kB_T + 8192;        // P [r][j]
constexpr int kB_DP = kB_P + 8192;       // dP o Gam [r][j]
constexpr int kB_M = kB_DP + 8192;       // M = beta dA o Gam [r][j]
constexpr int kB_X = kB_M + 8192;        // three 16 KB slots, reused by phase
constexpr int kB_GATE = kB_X + 3 * 16384;  // gam, e, f, beta, db1, db2, dlc [64] each + red [4][64]
constexpr int kB_BAR = kB_GATE + 7 * 256 + 1024 + 64;
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
  const __nv_bfloat16* v;
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

// Sums v[0..63] over the 128 threads of the CTA; out[r] (r < 64) gets the sum.
// Within a warp: five halving exchange steps (lane l ends with the sums of
// indices 2l, 2l+1); across warps: red[4][64] in shared memory.
__device__ __forceinline__ void cta_sum64(float (&v)[64], float* red, float* out) {
  const int l = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int off = 16 >> step, half = 32 >> step;
    const bool up = (l & off) != 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < half) {
        const float send = up ? v[i] : v[i + half];
        const float keep = up ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
  }
  red[w * 64 + 2 * l] = v[0];
  red[w * 64 + 2 * l + 1] = v[1];
  __syncthreads();
  if (threadIdx.x < 64)
    out[threadIdx.x] = red[threadIdx.x] + red[64 + threadIdx.x] + red[128 + threadIdx.x] +
                       red[192 + threadIdx.x];
  __syncthreads();
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  float a[32];
  tmem_ld32(taddr, a);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = a[i];
  tmem_ld32(taddr + 32, a);
#pragma unroll
  for (int i = 0; i < 32; ++i) v[32 + i] = a[i];
}

__global__ void __launch_bounds__(NT, 1)
gdn_tc_bwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_do, BwdParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid / 32;
  const int bh = blockIdx.x, b = bh / p.H, h = bh % p.H;

  float* gam = reinterpret_cast<float*>(sm + kB_GATE);
  float* ee = gam + 64;
  float* ff = ee + 64;
  float* bt = ff + 64;
  float* db1 = bt + 64;
  float* db2 = db1 + 64;
  float* dlc = db2 + 64;
  float* red = dlc + 64;  // [4][64]
  float* eC = red + 256;
  uint64_t* bar_load = reinterpret_cast<uint64_t*>(sm + kB_BAR);
  uint64_t* bar_mma = bar_load + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mma + 1);
  float* Am = reinterpret_cast<float*>(sm + kB_X);
  float* Tm = Am + 64 * kLdA;
  float* Sm = Tm + 64 * kLdA;
  const uint32_t sKQ = smem_u32(sm + kB_KQ), sZO = smem_u32(sm + kB_ZO);
  const uint32_t sGI = smem_u32(sm + kB_GI), sDG = smem_u32(sm + kB_DG);
  const uint32_t sT = smem_u32(sm + kB_T), sP = smem_u32(sm + kB_P);
  const uint32_t sDP = smem_u32(sm + kB_DP), sM = smem_u32(sm + kB_M);
  const uint32_t sX0 = smem_u32(sm + kB_X), sX1 = sX0 + 16384, sX2 = sX0 + 32768;

  if (tid == 0) {
    mbar_init(bar_load, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_do);
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kTmCols);
    tmem_relinquish();
  }
  cta_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lb = (uint32_t)(warp * 32) << 16;

  float dG[D];
#pragma unroll
  for (int d = 0; d < D; ++d) dG[d] = p.dht ? p.dht[((size_t)bh * D + d) * D + tid] : 0.f;
  store_g_tile(sm + kB_DG, dG, tid, nullptr);
  // <dH_out, H_out> of the chunk being processed (the last chunk: <dht, ht>)
  float carry = p.dht_dot ? p.dht_dot[bh] : 0.f;

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
      mbar_arrive_expect_tx(bar_load, 6 * 8192 + 32768);
      tma_load_4d(sm + kB_KQ + 0, &tm_k, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_KQ + 8192, &tm_q, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_KQ + 16384, &tm_k, bar_load, 64, h, t0, b);
      tma_load_4d(sm + kB_KQ + 24576, &tm_q, bar_load, 64, h, t0, b);
      tma_load_4d(sm + kB_ZO + 8192, &tm_do, bar_load, 0, h, t0, b);
      tma_load_4d(sm + kB_ZO + 24576, &tm_do, bar_load, 64, h, t0, b);
      bulk_load(sm + kB_GI, p.states + ((size_t)bh * p.N + ci) * 32768, 32768, bar_load);
    }
    // gates
    if (warp == 0) {
      const int l = tid;
      const size_t base = ((size_t)b * p.T + t0) * p.H + h;
      float g0 = l < n ? p.g[base + (size_t)l * p.H] : 0.f;
      float g1 = l + 32 < n ? p.g[base + (size_t)(l + 32) * p.H] : 0.f;
      bt[l] = l < n ? p.beta[base + (size_t)l * p.H] : 0.f;
      bt[l + 32] = l + 32 < n ? p.beta[base + (size_t)(l + 32) * p.H] : 0.f;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        float a0 = __shfl_up_sync(0xffffffffu, g0, off);
        float a1 = __shfl_up_sync(0xffffffffu, g1, off);
        if (l >= off) g0 += a0, g1 += a1;
      }
      g1 += __shfl_sync(0xffffffffu, g0, 31);
      const float gl = __shfl_sync(0xffffffffu, g1, 31);
      gam[l] = g0;
      gam[l + 32] = g1;
      ee[l] = expf(g0);
      ee[l + 32] = expf(g1);
      ff[l] = expf(gl - g0);
      ff[l + 32] = expf(gl - g1);
      if (l == 0) *eC = expf(gl);
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
      float kk[64];
      tmem_ld64(tmem + lb + kBtKQ, kk);
      if (tid < 64) {
        const int r = tid;
        const float gr = gam[r], br = bt[r];
#pragma unroll
        for (int j = 0; j < 64; ++j) Am[r * kLdA + j] = (j < r) ? br * kk[j] * expf(gr - gam[j]) : 0.f;
      } else {
        const int r = tid - 64;
        const float gr = gam[r];
#pragma unroll
        for (int j = 0; j < 64; ++j) kk[j] = (j <= r) ? kk[j] * expf(gr - gam[j]) : 0.f;
        store_row64(sm + kB_P, r, kk);
      }
    }
    cta_sync();
    solve_unit_lower(Am, Tm, Sm);
    {
      const int r = tid >> 1, hf = tid & 1;
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int j = hf * 32 + i;
        v[i] = (j <= r) ? Tm[r * kLdA + j] : 0.f;
      }
#pragma unroll
      for (int c8 = 0; c8 < 4; ++c8) {
        uint4 pk;
        uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          __nv_bfloat162 a = __floats2bfloat162_rn(v[c8 * 8 + 2 * i], v[c8 * 8 + 2 * i + 1]);
          w[i] = *reinterpret_cast<uint32_t*>(&a);
        }
        *reinterpret_cast<uint4*>(sm + kB_T + sw_row_off(r, hf * 4 + c8)) = pk;
      }
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
    // ---- E3: beta R^T -> X0, dU^T -> X1
    {
      float a[64], x[64];
      tmem_ld64(tmem + lb + kBtR, a);
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        const float vr = r < n ? __bfloat162float(p.v[(((size_t)b * p.T + t0 + r) * p.H + h) * D + tid]) : 0.f;
        a[r] = bt[r] * (vr + ee[r] * a[r]);
      }
      store_row64(sm + kB_X, tid, a);
      tmem_ld64(tmem + lb + kBtX1, a);
      tmem_ld64(tmem + lb + kBtX2, x);
#pragma unroll
      for (int j = 0; j < 64; ++j) a[j] = ff[j] * a[j] + x[j];
      store_row64(sm + kB_X + 16384, tid, a);
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
    float acc[64];  // per-lane terms of the log-gate gradient (summed over lanes later)
    {
      float u[64];
      tmem_ld64(tmem + lb + kBtU, u);
      store_row64(sm + kB_X, tid, u);
#pragma unroll
      for (int j = 0; j < 64; ++j) u[j] *= ff[j];
      store_row64(sm + kB_X + 32768, tid, u);
      float z[64], rr[64];
      tmem_ld64(tmem + lb + kBtZ, z);
      tmem_ld64(tmem + lb + kBtR, rr);
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        const size_t off = (((size_t)b * p.T + t0 + r) * p.H + h) * D + tid;
        const float vr = r < n ? __bfloat162float(p.v[off]) : 0.f;
        const float dr = bt[r] * z[r];
        if (r < n) p.dv[off] = __float2bfloat16_rn(dr);
        acc[r] = -vr * dr;                       // -v . dv
        rr[r] = z[r] * (vr + ee[r] * rr[r]);     // dZ_rc R_rc
        // dZ row r, column c = tid, into the dZ half of the [dZ; dO] operand
        const int half = tid >> 6, cc = tid & 63;
        *reinterpret_cast<__nv_bfloat16*>(sm + kB_ZO + half * 16384 + sw_row_off(r, cc >> 3) +
                                          (cc & 7) * 2) = __float2bfloat16_rn(z[r]);
        z[r] = ee[r] * dr;
      }
      store_row64(sm + kB_X + 16384, tid, z);
      cta_sum64(rr, red, db1);
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
      float x[64];
      tmem_ld64(tmem + lb + kBtX1, x);
      if (tid < 64) {
        // dA = -strict_lower(dZ U^T); dbeta part 2; M = beta dA o Gam
        const int r = tid;
        float kk[64];
        tmem_ld64(tmem + lb + kBtKQ, kk);
        const float gr = gam[r], br = bt[r];
        float s2 = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float w = (j < r) ? expf(gr - gam[j]) : 0.f;
          const float da = -x[j];
          s2 += da * kk[j] * w;
          x[j] = br * da * w;
        }
        db2[r] = s2;
        store_row64(sm + kB_M, r, x);
      } else {
        const int r = tid - 64;
        float kk[64];
        tmem_ld64(tmem + lb + kBtKQ, kk);  // keep the warp-collective load uniform
        const float gr = gam[r];
#pragma unroll
        for (int j = 0; j < 64; ++j) x[j] = (j <= r) ? x[j] * expf(gr - gam[j]) : 0.f;
        store_row64(sm + kB_DP, r, x);
      }
    }
    // scale dO rows by e in place (dO is done as an operand of dO^T P and G4)
    for (int i = tid; i < 2 * 64 * 8; i += NT) {
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
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        tmem_ld32(tmem + lb + kBtG3 + q4 * 32, v32);
#pragma unroll
        for (int i = 0; i < 32; ++i) dG[q4 * 32 + i] = fmaf(ec, dG[q4 * 32 + i], v32[i]);
      }
      float x[64];
      tmem_ld64(tmem + lb + kBtX2, x);  // dQ^T row d = tid
#pragma unroll
      for (int r = 0; r < 64; ++r) {
        const size_t off = (((size_t)b * p.T + t0 + r) * p.H + h) * D + tid;
        // q from the K|Q tile: row r, column d = tid
        const int half = tid >> 6, cc = tid & 63;
        const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
            sm + kB_KQ + half * 16384 + 8192 + sw_row_off(r, cc >> 3) + (cc & 7) * 2));
        acc[r] += qv * x[r];
        if (r < n) p.dq[off] = __float2bfloat16_rn(x[r]);
      }
      tmem_ld64(tmem + lb + kBtU, x);  // dK^T row d = tid
#pragma unroll
      for (int j = 0; j < 64; ++j)
        if (j < n) p.dk[(((size_t)b * p.T + t0 + j) * p.H + h) * D + tid] = __float2bfloat16_rn(x[j]);
    }
    cta_sum64(acc, red, dlc);
    if (tid < 64) {
      const int r = tid;
      if (r < n) p.dbeta[((size_t)b * p.T + t0 + r) * p.H + h] = db1[r] + db2[r];
    }
    // <dH_in, H_in> of this chunk = <dH_out, H_out> of the chunk before it
    float dot = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 pk = *reinterpret_cast<const uint4*>(sm + kB_GI + half * 16384 + sw_row_off(tid, c8));
        const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&pk);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float2 f2 = __bfloat1622float2(h2[i]);
          dot = fmaf(dG[half * 64 + c8 * 8 + 2 * i], f2.x, dot);
          dot = fmaf(dG[half * 64 + c8 * 8 + 2 * i + 1], f2.y, dot);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if ((tid & 31) == 0) red[warp] = dot;
    __syncthreads();
    if (warp == 0) {
      // dg_t = sum_{s >= t, s in chunk} (q_s.dq_s - v_s.dv_s) + <dH_out, H_out>
      float a0 = dlc[tid], a1 = dlc[tid + 32];
      float s1 = a1;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, s1, off);
        if (tid + off < 32) s1 += y;
      }
      const float tot1 = __shfl_sync(0xffffffffu, s1, 0);
      float s0 = a0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_down_sync(0xffffffffu, s0, off);
        if (tid + off < 32) s0 += y;
      }
      s0 += tot1;
      const size_t base = ((size_t)b * p.T + t0) * p.H + h;
      if (tid < n) p.dg[base + (size_t)tid * p.H] = carry + s0;
      if (tid + 32 < n) p.dg[base + (size_t)(tid + 32) * p.H] = carry + s1;
    }
    carry = red[0] + red[1] + red[2] + red[3];
    store_g_tile(sm + kB_DG, dG, tid, nullptr);
  }

  if (!ok) {
    if (tid == 0) report_timeout();
    mbar_wait(bar_load, load_phase, 1u << 20);
  } else if (p.dh0) {
#pragma unroll
    for (int d = 0; d < D; ++d) p.dh0[((size_t)bh * D + d) * D + tid] = dG[d];
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
  gdn_tc_fwd_kernel<<<p.B * p.H, NT, kSmemBytes, s>>>(mq, mk, mv, fp);
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
  CUtensorMap mq, mk, mdo;
  if ((e = make_token_map(&mq, p.q, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mk, p.k, p)) != cudaSuccess) return e;
  if ((e = make_token_map(&mdo, p.do_, p)) != cudaSuccess) return e;
  BwdParams bp{p.g, p.beta, static_cast<const __nv_bfloat16*>(p.v), p.dht, dht_dot,
               reinterpret_cast<const unsigned char*>(states), static_cast<__nv_bfloat16*>(p.dq),
               static_cast<__nv_bfloat16*>(p.dk_), static_cast<__nv_bfloat16*>(p.dv_), p.dg, p.dbeta,
               p.dh0, p.B, p.T, p.H, p.N};
  e = cudaFuncSetAttribute(gdn_tc_bwd_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kBwdSmemBytes);
  if (e != cudaSuccess) return e;
  prof_before(s);
  gdn_tc_bwd_kernel<<<p.B * p.H, NT, kBwdSmemBytes, s>>>(mq, mk, mdo, bp);
  prof_after(s, kTcBwd);
  return cudaGetLastError();
}

}  // namespace gdn
