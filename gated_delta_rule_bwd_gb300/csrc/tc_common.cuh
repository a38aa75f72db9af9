// Building blocks shared by the tensor-core kernel files (GDN and KDA):
// shared-memory tile layout helpers, bulk copies, the blocked 64 x 64
// unit-lower-triangular solve, cross-thread reductions, the per-file device
// status word of the bounded waits, and the host-side tensor-map / launch
// helpers.  Tiles are the 128-byte-swizzled K-major layouts described in
// tc_ptx.cuh.
#pragma once

#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "gdn.h"
#include "gdn_internal.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace tc {

// Status word of the bounded device-side waits of the kernels in the file
// that includes this header (each file has its own copy).
static __device__ int g_file_status = 0;

__device__ __forceinline__ void report_timeout() { atomicExch(&g_file_status, GDN_ERR_DEVICE_TIMEOUT); }

// Reads and clears this file's status word on the current device.
static inline cudaError_t read_and_clear_file_status(int* status) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_file_status, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbol(g_file_status, &zero, sizeof(int));
  if (e != cudaSuccess) return e;
  *status = v;
  return cudaSuccess;
}

constexpr int C = 64;     // chunk
constexpr int D = 128;    // dk = dv

constexpr int kLdF = 68;                   // fp32 row stride of A and T in the solve (16-byte rows)
constexpr int kSolveScratch = 32 * 36;     // largest solve scratch use: the 32 x 32 product, row stride 36
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

// 1-D bulk copy global -> shared completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16)
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy shared -> global (bulk-group completion; same alignment rules)
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_u32(src)), "r"(bytes)
               : "memory");
}

constexpr int kGroup = 256;
constexpr int kBarChain = 1, kBarPrep = 2;

// 64-element row chunk helper: writes nchunks groups of 8 bf16 (16 B) of a
// swizzled 128-byte row, starting at 16-byte chunk c0 (and the same bytes to
// dst if given).
__device__ __forceinline__ void store_chunks(unsigned char* tile, int row, int c0, const float* v,
                                             int nchunks, unsigned char* dst = nullptr) {
  for (int k = 0; k < nchunks; ++k) {
    uint4 pk;
    uint32_t* w = reinterpret_cast<uint32_t*>(&pk);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b2 = __floats2bfloat162_rn(v[k * 8 + 2 * i], v[k * 8 + 2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t*>(&b2);
    }
    const int off = sw_row_off(row, c0 + k);
    *reinterpret_cast<uint4*>(tile + off) = pk;
    if (dst) *reinterpret_cast<uint4*>(dst + off) = pk;
  }
}

// Scales each 128-byte bf16 row r of `rows` consecutive rows by s[r]
// (16-byte chunks spread over nth threads; t = this thread's index).
__device__ __forceinline__ void scale_rows(unsigned char* base, int rows, const float* s, int t,
                                           int nth) {
  for (int i = t; i < rows * 8; i += nth) {
    const int r = i >> 3;
    uint4* ptr = reinterpret_cast<uint4*>(base + i * 16);
    uint4 val = *ptr;
    __nv_bfloat162* h2 = reinterpret_cast<__nv_bfloat162*>(&val);
    const float e = s[r];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      float2 f2 = __bfloat1622float2(h2[k]);
      h2[k] = __floats2bfloat162_rn(f2.x * e, f2.y * e);
    }
    *ptr = val;
  }
}

// ---- small fp32 products on the warp-level tensor path (TF32, fp32 accumulate)
// used by the 64 x 64 triangular solve.  Fragment layout of mma.m16n8k8:
// g = lane / 4, q = lane % 4; A (16 x 8, row-major) a0 = A[g][q], a1 = A[g+8][q],
// a2 = A[g][q+4], a3 = A[g+8][q+4]; B (8 x 8) b0 = B[q][g], b1 = B[q+4][g];
// C (16 x 8) c0 = C[g][2q], c1 = C[g][2q+1], c2 = C[g+8][2q], c3 = C[g+8][2q+1].
// Row strides of 68, 36 or 24 floats make these loads conflict-free.

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

// d += A[m0:m0+16][ka:ka+8] * B[kb:kb+8][n0:n0+8]
__device__ __forceinline__ void tf32_mma_step(float (&d)[4], const float* A, int lda, int m0, int ka,
                                              const float* B, int ldb, int kb, int n0) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const uint32_t a0 = to_tf32(A[(m0 + g) * lda + ka + q]);
  const uint32_t a1 = to_tf32(A[(m0 + g + 8) * lda + ka + q]);
  const uint32_t a2 = to_tf32(A[(m0 + g) * lda + ka + q + 4]);
  const uint32_t a3 = to_tf32(A[(m0 + g + 8) * lda + ka + q + 4]);
  const uint32_t b0 = to_tf32(B[(kb + q) * ldb + n0 + g]);
  const uint32_t b1 = to_tf32(B[(kb + q + 4) * ldb + n0 + g]);
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void store_c_tile(const float (&d)[4], float* C, int ldc, int m0, int n0) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  *reinterpret_cast<float2*>(C + (m0 + g) * ldc + n0 + 2 * q) = make_float2(d[0], d[1]);
  *reinterpret_cast<float2*>(C + (m0 + g + 8) * ldc + n0 + 2 * q) = make_float2(d[2], d[3]);
}

// T = (I + A)^-1 for a 64 x 64 strictly lower A (fp32, row stride kLdF).  T
// is valid on and below the diagonal; above it only the entries that the
// steps read are zeroed, so callers mask columns j > r.  Three steps:
//  1. each 16 x 16 diagonal block by one warp: its two 8 x 8 diagonal blocks
//     by forward substitution (one lane per column), then the 8 x 8 coupling
//     T21 = -T22 (A21 T11);
//  2. inside each 32 x 32 half, T[1][0] = -T[1][1] (A[1][0] T[0][0]) over the
//     16 x 16 blocks (and the same for blocks 3, 2);
//  3. T_BA = -T_B (A_BA T_A) for the 32 x 32 halves.
// Steps 2 and 3 run on the warp-level tensor path in TF32 with fp32
// accumulation (its rounding is below that of the bf16 copies of T made next).
// nth threads take part (t = this thread's index, nth >= 256); sync() is
// their barrier.  S holds kSolveScratch floats (step 1 uses S[0, 256), step 2
// S[256, 1024), step 3 S[0, 32 * 36)).
template <class Sync>
__device__ void solve_unit_lower(const float* A, float* T, float* S, int t, int nth, Sync sync) {
  const int w = t >> 5, l = t & 31;
  if (w < 4) {
    const int o = w * 16;
    if (l < 16) {
      const int so = o + (l >> 3) * 8, jj = l & 7;
      float x[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float4 a0 = *reinterpret_cast<const float4*>(A + (so + r) * kLdF + so);
        const float4 a1 = *reinterpret_cast<const float4*>(A + (so + r) * kLdF + so + 4);
        const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int i = 0; i < r; ++i) {
          if (i & 1) s1 = fmaf(a[i], x[i], s1);
          else s0 = fmaf(a[i], x[i], s0);
        }
        x[r] = (r == jj) ? 1.f : ((r > jj) ? -(s0 + s1) : 0.f);
      }
#pragma unroll
      for (int r = 0; r < 8; ++r) T[(so + r) * kLdF + so + jj] = x[r];
    } else {
      // zero the 8 x 8 block above the diagonal of this 16 x 16 block
      for (int i = l - 16; i < 64; i += 16) T[(o + (i >> 3)) * kLdF + o + 8 + (i & 7)] = 0.f;
    }
    __syncwarp();
    float* S8 = S + w * 64;
    const int r = l >> 2, c = (l & 3) * 2;
    {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float a = A[(o + 8 + r) * kLdF + o + k];
        s0 = fmaf(a, T[(o + k) * kLdF + o + c], s0);
        s1 = fmaf(a, T[(o + k) * kLdF + o + c + 1], s1);
      }
      S8[r * 8 + c] = s0;
      S8[r * 8 + c + 1] = s1;
    }
    __syncwarp();
    {
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float a = T[(o + 8 + r) * kLdF + o + 8 + k];  // zero for k > r
        s0 = fmaf(a, S8[k * 8 + c], s0);
        s1 = fmaf(a, S8[k * 8 + c + 1], s1);
      }
      T[(o + 8 + r) * kLdF + o + c] = -s0;
      T[(o + 8 + r) * kLdF + o + c + 1] = -s1;
    }
  } else if (t < 256) {
    // zero the two 16 x 16 blocks above the block diagonal that steps 2 and 3
    // read as operands: rows 0-15 x columns 16-31 and rows 32-47 x columns 48-63
    const int i = t - 128, blk = i >> 6, rr = (i >> 2) & 15, c4 = (i & 3) * 4;
    *reinterpret_cast<float4*>(T + (32 * blk + rr) * kLdF + 32 * blk + 16 + c4) =
        make_float4(0.f, 0.f, 0.f, 0.f);
  }
  sync();
  // step 2: per 32 x 32 half b, S = A[2b+1][2b] T[2b][2b], T[2b+1][2b] = -T[2b+1][2b+1] S
  // (16 x 16 blocks); warp w < 4 takes half w / 2 and output columns 8 (w % 2) + [0, 8)
  if (w < 4) {
    const int hb = w >> 1, n0 = (w & 1) * 8;
    const int r0 = 32 * hb + 16, c0 = 32 * hb;
    float* Sb = S + 256 + hb * 16 * 24;  // 16 x 16, row stride 24
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) tf32_mma_step(d, A, kLdF, r0, c0 + k0, T, kLdF, c0 + k0, c0 + n0);
    store_c_tile(d, Sb, 24, 0, n0);
    __syncwarp();  // this warp's columns of S are all it reads next
    float e[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 16; k0 += 8) tf32_mma_step(e, T, kLdF, r0, r0 + k0, Sb, 24, k0, n0);
#pragma unroll
    for (int i = 0; i < 4; ++i) e[i] = -e[i];
    store_c_tile(e, T, kLdF, r0, c0 + n0);
  }
  sync();
  // step 3: S32 = A[32:64][0:32] T[0:32][0:32], T[32:64][0:32] = -T[32:64][32:64] S32;
  // 8 output tiles of 16 x 8 (warp w < 8 takes tile w)
  if (w < 8) {
    const int m0 = (w >> 2) * 16, n0 = (w & 3) * 8;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) tf32_mma_step(d, A, kLdF, 32 + m0, k0, T, kLdF, k0, n0);
    store_c_tile(d, S, 36, m0, n0);
  }
  sync();
  if (w < 8) {
    const int m0 = (w >> 2) * 16, n0 = (w & 3) * 8;
    float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k0 = 0; k0 < 32; k0 += 8) tf32_mma_step(d, T, kLdF, 32 + m0, 32 + k0, S, 36, k0, n0);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = -d[i];
    store_c_tile(d, T, kLdF, 32 + m0, n0);
  }
  sync();
}

__device__ __forceinline__ void group_sync_tc(int id) {
  tc_fence_before();
  group_sync(id, kGroup);
  tc_fence_after();
}

// n-column form of cta_sum_rows16 for any CTA of 128 x (64 / n) threads:
// each thread holds v[i] for tile column (n cg + i) of its row (cg = warp / 4);
// out[r] (r < 64) gets the sum over all 128 rows.  Within a warp log2(n)
// halving exchanges leave lane l with column n cg + (l >> (5 - log2 n)),
// summed over the lanes that differ in the low bits by the remaining xor
// adds; across the four warps of a column group via red[(4 cg + quad) n + i].
template <int n>
__device__ __forceinline__ void cta_sum_rows(float (&v)[n], float* red, float* out) {
  constexpr int steps = n == 16 ? 4 : n == 8 ? 3 : n == 4 ? 2 : 1;
  const int l = threadIdx.x & 31, w = threadIdx.x >> 5, quad = w & 3, cg = w >> 2;
#pragma unroll
  for (int step = 0; step < steps; ++step) {
    const int off = 16 >> step, half = (n / 2) >> step;
    const bool up = (l & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      if (i < half) {
        const float send = up ? v[i] : v[i + half];
        const float keep = up ? v[i + half] : v[i];
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
      }
    }
  }
#pragma unroll
  for (int off = 16 >> steps; off > 0; off >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
  constexpr int sh = 5 - steps;
  if ((l & ((1 << sh) - 1)) == 0) red[(cg * 4 + quad) * n + (l >> sh)] = v[0];
  __syncthreads();
  if (threadIdx.x < 64) {
    const int c = threadIdx.x / n, i = threadIdx.x % n;
    out[threadIdx.x] = red[(c * 4 + 0) * n + i] + red[(c * 4 + 1) * n + i] +
                       red[(c * 4 + 2) * n + i] + red[(c * 4 + 3) * n + i];
  }
  __syncthreads();
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

// Writes x as the bf16 element (token r, feature d) of a [64 x 128] staging tile
// made of two K-major 128-byte-swizzled halves (features 0-63, 64-127; 8 KB
// each) -- the layout a TMA store of two 64 x 64 boxes reads.
__device__ __forceinline__ void stage_bf16(unsigned char* tile2, int r, int d, float x) {
  *reinterpret_cast<__nv_bfloat16*>(tile2 + (d >> 6) * 8192 + sw_row_off(r, (d & 63) >> 3) +
                                    (d & 7) * 2) = __float2bfloat16_rn(x);
}

// Stages a warp's 32 x 16 block of a transposed tile -- TMEM lanes (features)
// lane0 .. lane0 + 31, columns (tokens) col0 .. col0 + 15 -- as bf16 rows of a
// [64 x 128] token-major staging tile made of two K-major 128-byte-swizzled
// feature halves `half_stride` bytes apart (element (token r, feature d) at
// tile2 + (d >> 6) half_stride + sw_row_off(r, (d & 63) >> 3) + (d & 7) 2),
// with f(token, value) applied first: two 16x256b loads and two transposed
// 4-matrix stores per 16 lanes instead of one scalar store per element.
// With tmem_b (and tmem_c) != 0 the staged value is the sum of the TMEM blocks.
template <typename F>
__device__ __forceinline__ void stage_tmem_block(unsigned char* tile2, int half_stride,
                                                 uint32_t tmem_lane0_col0, int lane0, int col0,
                                                 F f, uint32_t tmem_b = 0, uint32_t tmem_c = 0) {
  const int t = threadIdx.x & 31;
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    float v[8];
    tmem_ld16x16(tmem_lane0_col0 + ((uint32_t)(16 * hh) << 16), v);
    if (tmem_b) {
      float u[8];
      tmem_ld16x16(tmem_b + ((uint32_t)(16 * hh) << 16), u);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += u[i];
    }
    if (tmem_c) {
      float u[8];
      tmem_ld16x16(tmem_c + ((uint32_t)(16 * hh) << 16), u);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += u[i];
    }
    const int f0 = lane0 + 16 * hh;  // first feature of these 16 lanes
    const int c = col0 + 2 * (t & 3);
    uint32_t w[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {  // matrix m: features f0 + 8 (m & 1), tokens col0 + 8 (m >> 1)
      const int tok = c + 8 * (m >> 1);
      __nv_bfloat162 b2 = __floats2bfloat162_rn(f(tok, v[2 * m]), f(tok + 1, v[2 * m + 1]));
      w[m] = *reinterpret_cast<uint32_t*>(&b2);
    }
    // this thread's row address: matrix t / 8, stored row t % 8
    const int m = t >> 3, tok = col0 + 8 * (m >> 1) + (t & 7), fe = f0 + 8 * (m & 1);
    unsigned char* dst = tile2 + (fe >> 6) * half_stride + sw_row_off(tok, (fe & 63) >> 3);
    stmatrix_x4_trans(smem_u32(dst), w[0], w[1], w[2], w[3]);
  }
}

// Writes rows [0, n) of a [64 x 128] bf16 staging tile (two K-major
// 128-byte-swizzled halves of 8 KB, features 0-63 and 64-127) to global rows
// dst + r * row_stride (in elements), 16 bytes per store; t / nth: this
// thread's index among nth writers.  Used for a packed sequence's last
// chunk, whose rows past the sequence belong to the next one (a tensor store
// would write all 64).
__device__ __forceinline__ void store_rows_bf16(const unsigned char* tile2, __nv_bfloat16* dst,
                                                size_t row_stride, int n, int t, int nth) {
  for (int i = t; i < n * 16; i += nth) {
    const int r = i >> 4, hh = (i >> 3) & 1, c8 = i & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(tile2 + hh * 8192 + sw_row_off(r, c8));
    *reinterpret_cast<uint4*>(dst + r * row_stride + hh * 64 + c8 * 8) = v;
  }
}

// bf16 element (row, col) of a swizzled 64-wide K-major tile
__device__ __forceinline__ float tile_elem(const unsigned char* tile, int row, int col) {
  return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
      tile + sw_row_off(row, col >> 3) + (col & 7) * 2));
}


// ---------------------------------------------------------------- host side

inline PFN_cuTensorMapEncodeTiled_v12000 get_encoder() {
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
inline cudaError_t make_token_map(CUtensorMap* m, const void* ptr, const Problem& p) {
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

// Launches a kernel that may start while the previous kernel in the stream
// finishes (programmatic stream serialization): the kernels of this file wait
// for it with grid_dep_wait() after their prologue (barrier set-up, TMEM
// allocation) and before any global-memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), unsigned grid, unsigned block,
                              size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  return n;
}


}  // namespace tc
}  // namespace gdn
