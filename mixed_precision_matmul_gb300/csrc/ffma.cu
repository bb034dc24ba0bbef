// Plain fp32 CUDA-core product, the comparator of the split-precision modes:
// every output element is ONE sequential fmaf chain over k in ascending
// order, acc = fmaf(a(i,k), b(k,j), acc), followed by
// out = fmaf(beta, C, alpha * acc).  This is the "fp32 has no MMA instruction,
// so it stays FFMA-bound" path of "tile_matmul(): use the cuBLASDx
// register-accumulator API ...", spike results, second bullet.
//
// Tiling: 128 x 128 output tile per 256-thread block, k-tiles of 8 staged in
// shared memory (double buffered, prefetched through registers), 8 x 8
// outputs per thread in registers.  Any layout, leading dimension and tail.
#include "internal.h"

namespace mpg {
namespace {

constexpr int kBM = 128, kBN = 128, kBK = 8, kThreads = 256;
constexpr int kPad = 4;

struct FfmaTileLoader {
  // each thread loads 4 elements of the A tile and 4 of the B tile
  __device__ static void load(const FfmaParams& p, const float* a, const float* b, int m0, int n0, int k0,
                              float (&ra)[4], float (&rb)[4]) {
    const int t = threadIdx.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int mm, kk;
      if (p.a_col_major) {  // (m, k) at k*lda + m: 128 consecutive m per k
        mm = t & 127;
        kk = (t >> 7) + 2 * e;
      } else {              // (m, k) at m*lda + k: 8 consecutive k per m
        kk = t & 7;
        mm = (t >> 3) + 32 * e;
      }
      const int gm = m0 + mm, gk = k0 + kk;
      float v = 0.0f;
      if (gm < p.m && gk < p.k) v = p.a_col_major ? __ldg(a + (int64_t)gk * p.lda + gm) : __ldg(a + (int64_t)gm * p.lda + gk);
      ra[e] = v;
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      int nn, kk;
      if (p.b_col_major) {  // (k, n) at n*ldb + k
        kk = t & 7;
        nn = (t >> 3) + 32 * e;
      } else {              // (k, n) at k*ldb + n
        nn = t & 127;
        kk = (t >> 7) + 2 * e;
      }
      const int gn = n0 + nn, gk = k0 + kk;
      float v = 0.0f;
      if (gn < p.n && gk < p.k) v = p.b_col_major ? __ldg(b + (int64_t)gn * p.ldb + gk) : __ldg(b + (int64_t)gk * p.ldb + gn);
      rb[e] = v;
    }
  }
  __device__ static void store(const FfmaParams& p, float (*As)[kBM + kPad], float (*Bs)[kBN + kPad],
                               const float (&ra)[4], const float (&rb)[4]) {
    const int t = threadIdx.x;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (p.a_col_major) As[(t >> 7) + 2 * e][t & 127] = ra[e];
      else As[t & 7][(t >> 3) + 32 * e] = ra[e];
      if (p.b_col_major) Bs[t & 7][(t >> 3) + 32 * e] = rb[e];
      else Bs[(t >> 7) + 2 * e][t & 127] = rb[e];
    }
  }
};

__global__ void __launch_bounds__(kThreads, 2) ffma_gemm_kernel(const FfmaParams p) {
  __shared__ __align__(16) float As[2][kBK][kBM + kPad];
  __shared__ __align__(16) float Bs[2][kBK][kBN + kPad];
  const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * kBN;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int bz = blockIdx.z; bz < p.batch; bz += gridDim.z) {
    const float* a = p.a + (int64_t)bz * p.stride_a;
    const float* b = p.b + (int64_t)bz * p.stride_b;
    float* c = p.c + (int64_t)bz * p.stride_c;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;

    float ra[4], rb[4];
    const int num_kt = (p.k + kBK - 1) / kBK;
    FfmaTileLoader::load(p, a, b, m0, n0, 0, ra, rb);
    FfmaTileLoader::store(p, As[0], Bs[0], ra, rb);
    __syncthreads();
    for (int kt = 0; kt < num_kt; ++kt) {
      const int cur = kt & 1;
      if (kt + 1 < num_kt) FfmaTileLoader::load(p, a, b, m0, n0, (kt + 1) * kBK, ra, rb);
#pragma unroll
      for (int kk = 0; kk < kBK; ++kk) {
        const float4 a0 = *reinterpret_cast<const float4*>(&As[cur][kk][ty * 4]);
        const float4 a1 = *reinterpret_cast<const float4*>(&As[cur][kk][64 + ty * 4]);
        const float4 b0 = *reinterpret_cast<const float4*>(&Bs[cur][kk][tx * 4]);
        const float4 b1 = *reinterpret_cast<const float4*>(&Bs[cur][kk][64 + tx * 4]);
        const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
      }
      if (kt + 1 < num_kt) FfmaTileLoader::store(p, As[cur ^ 1], Bs[cur ^ 1], ra, rb);
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
        float* dst = c + (int64_t)gm * p.ldc + gn;
        *dst = (p.beta != 0.0f) ? fmaf(p.beta, *dst, p.alpha * acc[i][j]) : p.alpha * acc[i][j];
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_ffma(const FfmaParams& p, cudaStream_t stream) {
  dim3 grid((p.n + kBN - 1) / kBN, (p.m + kBM - 1) / kBM, p.batch < 65535 ? p.batch : 65535);
  ffma_gemm_kernel<<<grid, kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mpg
