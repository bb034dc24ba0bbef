// Small kernels around the main product: the device status word, C = beta*C
// (k == 0 or alpha == 0), the split-K reduction, the mma.sync m16n8k16
// accumulator-layout probe, the epilogue-staging probe and the bounded-wait
// self test.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "outio.cuh"
#include "ptx.cuh"
#include "staging.cuh"

namespace mpg {

// One status word per device (a module global: every device that loads the
// library holds its own copy).
__device__ uint32_t g_status_word;

uint32_t* status_word_ptr() {
  void* ptr = nullptr;
  if (cudaGetSymbolAddress(&ptr, g_status_word) != cudaSuccess) return nullptr;
  return static_cast<uint32_t*>(ptr);
}

namespace {

__global__ void scale_c_kernel(void* c, int c_dtype, int64_t ldc, int64_t stride_c, int32_t m, int32_t n,
                               int32_t batch, float beta) {
  const int64_t per = (int64_t)m * n;
  const int64_t total = per * batch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per;
    const int64_t r = (i - b * per) / n;
    const int64_t col = i - b * per - r * n;
    const int64_t idx = b * stride_c + r * ldc + col;
    out_store(c, idx, (beta != 0.0f) ? beta * out_load(c, idx, c_dtype) : 0.0f, c_dtype);
  }
}

// out = alpha * (partial[0] + partial[1] + ... ) + beta * C, partial sums
// added in split order.
__global__ void splitk_reduce_kernel(const float* __restrict__ partial, int32_t splits, void* c, int c_dtype,
                                     int64_t ldc, int64_t stride_c, int32_t m, int32_t n, int32_t batch,
                                     float alpha, float beta) {
  griddep_wait();   // launched as a programmatic dependent of the product that writes the partials
  const int64_t per = (int64_t)m * n;
  const int64_t total = per * batch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    float s = partial[i];
    for (int sp = 1; sp < splits; ++sp) s += partial[(int64_t)sp * total + i];
    const int64_t b = i / per;
    const int64_t r = (i - b * per) / n;
    const int64_t col = i - b * per - r * n;
    const int64_t idx = b * stride_c + r * ldc + col;
    out_store(c, idx, (beta != 0.0f) ? fmaf(beta, out_load(c, idx, c_dtype), alpha * s) : alpha * s, c_dtype);
  }
}

// One warp, one mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32.
// Operand fragments gathered per the PTX ISA layouts (groupID = lane/4,
// threadID_in_group = lane%4):
//   A (16x16 row): a0 = A[g][2t..2t+1], a1 = A[g+8][2t..], a2 = A[g][2t+8..], a3 = A[g+8][2t+8..]
//   B (16x8 col):  b0 = B[2t..2t+1][g], b1 = B[2t+8..2t+9][g]
// The accumulator fragment is written out unscattered: D[lane*4 + j].
__global__ void probe_mma_kernel(const unsigned short* __restrict__ A, const unsigned short* __restrict__ B,
                                 float* __restrict__ D) {
  const int lane = threadIdx.x;
  const int g = lane >> 2, t = lane & 3;
  auto pack = [](unsigned short lo, unsigned short hi) { return (uint32_t)lo | ((uint32_t)hi << 16); };
  const uint32_t a0 = pack(A[g * 16 + 2 * t], A[g * 16 + 2 * t + 1]);
  const uint32_t a1 = pack(A[(g + 8) * 16 + 2 * t], A[(g + 8) * 16 + 2 * t + 1]);
  const uint32_t a2 = pack(A[g * 16 + 2 * t + 8], A[g * 16 + 2 * t + 9]);
  const uint32_t a3 = pack(A[(g + 8) * 16 + 2 * t + 8], A[(g + 8) * 16 + 2 * t + 9]);
  // B column-major: element (k, n) at n*16 + k
  const uint32_t b0 = pack(B[g * 16 + 2 * t], B[g * 16 + 2 * t + 1]);
  const uint32_t b1 = pack(B[g * 16 + 2 * t + 8], B[g * 16 + 2 * t + 9]);
  float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  D[lane * 4 + 0] = d0;
  D[lane * 4 + 1] = d1;
  D[lane * 4 + 2] = d2;
  D[lane * 4 + 3] = d3;
}

// The same instruction with the fragments given verbatim per lane.
__global__ void probe_mma_frag_kernel(const uint32_t* __restrict__ Af, const uint32_t* __restrict__ Bf,
                                      float* __restrict__ D) {
  const int lane = threadIdx.x;
  const uint32_t a0 = Af[lane * 4], a1 = Af[lane * 4 + 1], a2 = Af[lane * 4 + 2], a3 = Af[lane * 4 + 3];
  const uint32_t b0 = Bf[lane * 2], b1 = Bf[lane * 2 + 1];
  float d0 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d0), "+f"(d1), "+f"(d2), "+f"(d3)
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  D[lane * 4 + 0] = d0;
  D[lane * 4 + 1] = d1;
  D[lane * 4 + 2] = d2;
  D[lane * 4 + 3] = d3;
}

// A single bounded wait on an mbarrier that nothing arrives at: the wait must
// expire, record the timeout in the status word and let the kernel return.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    WaitCtl c;
    c.abort = &abort_flag;
    c.status = status;
    c.limit_ns = limit_ns;
    (void)mbar_wait(&bar, 0, c);
  }
  __syncthreads();
}

int grid_for(int64_t total) {
  int64_t blocks = (total + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  return blocks < 1 ? 1 : (int)blocks;
}

}  // namespace

cudaError_t launch_scale_c(void* c, int c_dtype, int64_t ldc, int64_t stride_c, int32_t m, int32_t n,
                           int32_t batch, float beta, cudaStream_t stream) {
  scale_c_kernel<<<grid_for((int64_t)m * n * batch), 256, 0, stream>>>(c, c_dtype, ldc, stride_c, m, n, batch,
                                                                        beta);
  return cudaGetLastError();
}

cudaError_t launch_splitk_reduce(const float* partial, int32_t splits, void* c, int c_dtype, int64_t ldc,
                                 int64_t stride_c, int32_t m, int32_t n, int32_t batch, float alpha, float beta,
                                 cudaStream_t stream) {
  // a programmatic dependent of the product: it may be scheduled as the
  // product's CTAs finish and waits (griddep_wait) for all of their partials
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3((unsigned)grid_for((int64_t)m * n * batch));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, splitk_reduce_kernel, partial, splits, c, c_dtype, ldc, stride_c, m, n,
                                     batch, alpha, beta);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_probe_mma(const void* a, const void* b, float* d, cudaStream_t stream) {
  probe_mma_kernel<<<1, 32, 0, stream>>>(static_cast<const unsigned short*>(a),
                                         static_cast<const unsigned short*>(b), d);
  return cudaGetLastError();
}

cudaError_t launch_probe_mma_frag(const uint32_t* a, const uint32_t* b, float* d, cudaStream_t stream) {
  probe_mma_frag_kernel<<<1, 32, 0, stream>>>(a, b, d);
  return cudaGetLastError();
}

// Epilogue-staging probe: warp w of the grid moves blocks of 32 x 32 fp32
// (row-major, packed, 4 KB each) from `in` to `out` through its staging
// buffer exactly as the product epilogues do after tcgen05.ld: lane l holds
// row l and writes it, then the warp reads the block back by 16-byte chunks
// of rows (vector stores) or by columns (scalar stores).  Nothing else uses
// shared memory meanwhile, so the profiler's bank-conflict counters see the
// staging pattern alone.
__global__ void __launch_bounds__(256) probe_staging_kernel(const float* __restrict__ in, float* __restrict__ out,
                                                             int64_t blocks, int scalar) {
  __shared__ __align__(16) float stg_all[8][1024];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t stg = smem_addr(stg_all[warp]);
  for (int64_t b = (int64_t)blockIdx.x * 8 + warp; b < blocks; b += (int64_t)gridDim.x * 8) {
    const float* src = in + b * 1024;
    float* dst = out + b * 1024;
    float v[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float4 x = __ldg(reinterpret_cast<const float4*>(src + lane * 32 + 4 * c));
      v[4 * c] = x.x;
      v[4 * c + 1] = x.y;
      v[4 * c + 2] = x.z;
      v[4 * c + 3] = x.w;
    }
    stage_write_row(stg, lane, v);
    __syncwarp();
    if (!scalar) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int r = i * 4 + (lane >> 3);
        *reinterpret_cast<float4*>(dst + r * 32 + (lane & 7) * 4) = stage_read_chunk(stg, lane, i);
      }
    } else {
#pragma unroll 4
      for (int r = 0; r < 32; ++r) dst[r * 32 + lane] = stage_read_elem(stg, lane, r);
    }
    __syncwarp();
  }
}

cudaError_t launch_probe_staging(const float* in, float* out, int64_t blocks, int scalar, int sm_count,
                                 cudaStream_t stream) {
  const int64_t grid = std::min<int64_t>((blocks + 7) / 8, (int64_t)sm_count * 8);
  if (grid <= 0) return cudaSuccess;
  probe_staging_kernel<<<(unsigned)grid, 256, 0, stream>>>(in, out, blocks, scalar);
  return cudaGetLastError();
}

// Throughput probe of the fp32 multiply-add pipe, the bound of the FFMA
// comparator: every thread runs `iters` rounds of 32 independent fmaf chains
// (acc = fmaf(1, acc, 1), from acc = 0 .. 31), as scalar fmaf or as 16
// packed pairs (__ffma2_rn), with no memory traffic inside the loop.  The
// chains end at i + iters exactly, so thread 0 of each block writes
// 496 + 32 * iters, which checks that the work was done.
__global__ void __launch_bounds__(256) probe_fma_kernel(float* __restrict__ out, int iters, int packed, float a,
                                                         float b) {
  float s = 0.0f;
  if (packed) {
    float2 acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = make_float2((float)(2 * i), (float)(2 * i + 1));
    const float2 av = make_float2(a, a), bv = make_float2(b, b);
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = __ffma2_rn(av, acc[i], bv);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) s += acc[i].x + acc[i].y;
  } else {
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = (float)i;
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int i = 0; i < 32; ++i) acc[i] = fmaf(a, acc[i], b);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) s += acc[i];
  }
  if (threadIdx.x == 0) out[blockIdx.x] = s;
}

cudaError_t launch_probe_fma(float* out, int64_t blocks, int iters, int packed, cudaStream_t stream) {
  probe_fma_kernel<<<(unsigned)blocks, 256, 0, stream>>>(out, iters, packed, 1.0f, 1.0f);
  return cudaGetLastError();
}

cudaError_t launch_selftest_wait(uint32_t* status, uint64_t limit_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace mpg
