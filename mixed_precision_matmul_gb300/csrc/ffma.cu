// Plain fp32 CUDA-core product, the comparator of the split-precision modes:
// every output element is ONE sequential fmaf chain over k in ascending
// order, acc = fmaf(a(i,k), b(k,j), acc), followed by
// out = fmaf(beta, C, alpha * acc).  This is the "fp32 has no MMA instruction,
// so it stays FFMA-bound" path of "tile_matmul(): use the cuBLASDx
// register-accumulator API ...", spike results, second bullet.
//
// Tiling: 128 x 128 output tile per 256-thread block, k-tiles of 16 staged in
// shared memory (double buffered, prefetched through registers; A stored
// k-major so both operands are read as float4 broadcasts), 8 x 8 outputs per
// thread in registers.  Interior tiles of aligned operands load float4
// vectors; edge tiles and unaligned operands load element by element with
// bounds checks.  Any layout, leading dimension and tail.  The 64 chains of
// a thread advance two at a time with the packed fp32 FMA (__ffma2_rn: two
// independent correctly rounded fmaf in one instruction), which halves the
// issue slots the multiply-adds take and leaves each chain's steps unchanged.
#include "internal.h"
#include "outio.cuh"

namespace mpg {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 16, kThreads = 256;
constexpr int kPad = 4;

template <bool A_COL, bool B_COL>
struct Loader {
  // Each thread fetches 8 elements of the A tile and 8 of the B tile per k-tile.
  float ra[8], rb[8];

  __device__ void load(const FfmaParams& p, const float* a, const float* b, int m0, int n0, int k0, bool vec) {
    const int t = threadIdx.x;
    // ---- A (m x k)
    if (vec && m0 + kBM <= p.m && k0 + kBK <= p.k) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float4 v;
        if constexpr (A_COL) {  // m contiguous: 32 float4 per k line
          const int kk = (t >> 5) + 8 * i, mm = (t & 31) * 4;
          v = __ldg(reinterpret_cast<const float4*>(a + (int64_t)(k0 + kk) * p.lda + m0 + mm));
        } else {                // k contiguous: 4 float4 per row
          const int mm = (t >> 2) + 64 * i, kk = (t & 3) * 4;
          v = __ldg(reinterpret_cast<const float4*>(a + (int64_t)(m0 + mm) * p.lda + k0 + kk));
        }
        ra[4 * i] = v.x; ra[4 * i + 1] = v.y; ra[4 * i + 2] = v.z; ra[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          int mm, kk;
          if constexpr (A_COL) { kk = (t >> 5) + 8 * i; mm = (t & 31) * 4 + e; }
          else { mm = (t >> 2) + 64 * i; kk = (t & 3) * 4 + e; }
          const int gm = m0 + mm, gk = k0 + kk;
          float v = 0.0f;
          if (gm < p.m && gk < p.k)
            v = A_COL ? __ldg(a + (int64_t)gk * p.lda + gm) : __ldg(a + (int64_t)gm * p.lda + gk);
          ra[4 * i + e] = v;
        }
    }
    // ---- B (k x n)
    if (vec && n0 + kBN <= p.n && k0 + kBK <= p.k) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        float4 v;
        if constexpr (B_COL) {  // k contiguous: 4 float4 per column
          const int nn = (t >> 2) + 64 * i, kk = (t & 3) * 4;
          v = __ldg(reinterpret_cast<const float4*>(b + (int64_t)(n0 + nn) * p.ldb + k0 + kk));
        } else {                // n contiguous: 32 float4 per k line
          const int kk = (t >> 5) + 8 * i, nn = (t & 31) * 4;
          v = __ldg(reinterpret_cast<const float4*>(b + (int64_t)(k0 + kk) * p.ldb + n0 + nn));
        }
        rb[4 * i] = v.x; rb[4 * i + 1] = v.y; rb[4 * i + 2] = v.z; rb[4 * i + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          int nn, kk;
          if constexpr (B_COL) { nn = (t >> 2) + 64 * i; kk = (t & 3) * 4 + e; }
          else { kk = (t >> 5) + 8 * i; nn = (t & 31) * 4 + e; }
          const int gn = n0 + nn, gk = k0 + kk;
          float v = 0.0f;
          if (gn < p.n && gk < p.k)
            v = B_COL ? __ldg(b + (int64_t)gn * p.ldb + gk) : __ldg(b + (int64_t)gk * p.ldb + gn);
          rb[4 * i + e] = v;
        }
    }
  }

  // shared tiles are k-major: As[k][m], Bs[k][n]
  __device__ void store(float (*As)[kBM + kPad], float (*Bs)[kBN + kPad]) const {
    const int t = threadIdx.x;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      if constexpr (A_COL) {
        const int kk = (t >> 5) + 8 * i, mm = (t & 31) * 4;
        *reinterpret_cast<float4*>(&As[kk][mm]) = make_float4(ra[4 * i], ra[4 * i + 1], ra[4 * i + 2], ra[4 * i + 3]);
      } else {
        const int mm = (t >> 2) + 64 * i, kk = (t & 3) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) As[kk + e][mm] = ra[4 * i + e];
      }
      if constexpr (B_COL) {
        const int nn = (t >> 2) + 64 * i, kk = (t & 3) * 4;
#pragma unroll
        for (int e = 0; e < 4; ++e) Bs[kk + e][nn] = rb[4 * i + e];
      } else {
        const int kk = (t >> 5) + 8 * i, nn = (t & 31) * 4;
        *reinterpret_cast<float4*>(&Bs[kk][nn]) = make_float4(rb[4 * i], rb[4 * i + 1], rb[4 * i + 2], rb[4 * i + 3]);
      }
    }
  }
};

template <bool A_COL, bool B_COL>
__global__ void __launch_bounds__(kThreads, 2) ffma_gemm_kernel(const FfmaParams p, int a_vec, int b_vec) {
  __shared__ __align__(16) float As[2][kBK][kBM + kPad];
  __shared__ __align__(16) float Bs[2][kBK][kBN + kPad];
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const bool vec = a_vec && b_vec;
  for (int bz = blockIdx.z; bz < p.batch; bz += gridDim.z) {
    const float* a = p.a + (int64_t)bz * p.stride_a;
    const float* b = p.b + (int64_t)bz * p.stride_b;
    void* c = static_cast<uint8_t*>(p.c) + (int64_t)bz * p.stride_c * (p.c_dtype == kOutF32 ? 4 : 2);
    // acc[i][j] holds columns 2j and 2j+1 of row i: one packed fp32 FMA
    // (two independent correctly rounded fmaf) per pair
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    Loader<A_COL, B_COL> ld;
    const int num_kt = (p.k + kBK - 1) / kBK;
    ld.load(p, a, b, m0, n0, 0, vec);
    ld.store(As[0], Bs[0]);
    __syncthreads();
    for (int kt = 0; kt < num_kt; ++kt) {
      const int cur = kt & 1;
      if (kt + 1 < num_kt) ld.load(p, a, b, m0, n0, (kt + 1) * kBK, vec);
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) {
        const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][kk][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][kk][64 + tx * 4]);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float2 bv[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                              make_float2(b1.z, b1.w)};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float2 ai = make_float2(av[i], av[i]);
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, bv[j], acc[i][j]);
        }
      }
      if (kt + 1 < num_kt) ld.store(As[cur ^ 1], Bs[cur ^ 1]);
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int gm = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
      if (gm >= p.m) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int gn = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + (j - 4));
        if (gn >= p.n) continue;
        const int64_t idx = (int64_t)gm * p.ldc + gn;
        const float t = p.alpha * ((j & 1) ? acc[i][j >> 1].y : acc[i][j >> 1].x);
        out_store(c, idx, (p.beta != 0.0f) ? fmaf(p.beta, out_load(c, idx, p.c_dtype), t) : t, p.c_dtype);
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_ffma(const FfmaParams& p, cudaStream_t stream) {
  // float4 loads need 16-byte aligned bases, leading dimensions and batch strides
  auto aligned = [&](const float* x, int64_t ld, int64_t stride) {
    return reinterpret_cast<uintptr_t>(x) % 16 == 0 && ld % 4 == 0 && (p.batch == 1 || stride % 4 == 0);
  };
  // Rows in slices of at most 65535 tile rows (the grid's y limit): each
  // slice is the same product on A's and C's rows from its first row on.
  constexpr int64_t kSliceRows = (int64_t)65535 * kBM;
  const int64_t c_es = (p.c_dtype == kOutF32) ? 4 : 2;
  for (int64_t r0 = 0; r0 < p.m; r0 += kSliceRows) {
    FfmaParams q = p;
    q.m = (int32_t)(p.m - r0 < kSliceRows ? p.m - r0 : kSliceRows);
    q.a = p.a + (p.a_col_major ? r0 : r0 * p.lda);
    q.c = static_cast<uint8_t*>(p.c) + r0 * p.ldc * c_es;
    dim3 grid((unsigned)(((int64_t)q.n + kBN - 1) / kBN), (unsigned)((q.m + kBM - 1) / kBM),
              q.batch < 65535 ? q.batch : 65535);
    const int av = aligned(q.a, q.lda, q.stride_a), bv = aligned(q.b, q.ldb, q.stride_b);
    if (q.a_col_major && q.b_col_major) ffma_gemm_kernel<true, true><<<grid, kThreads, 0, stream>>>(q, av, bv);
    else if (q.a_col_major) ffma_gemm_kernel<true, false><<<grid, kThreads, 0, stream>>>(q, av, bv);
    else if (q.b_col_major) ffma_gemm_kernel<false, true><<<grid, kThreads, 0, stream>>>(q, av, bv);
    else ffma_gemm_kernel<false, false><<<grid, kThreads, 0, stream>>>(q, av, bv);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace mpg
