// Separate conversion pass of the fp32 operands: fp32 -> fp16 / bf16
// (round to nearest even) or the fp16 hi/lo split, written as packed 16-bit
// copies that the direct TMA path then multiplies.  The arithmetic is the
// converter warps' (same conversions, same split), so both routes give the
// same operands; this one trades one extra read and write of the operands in
// HBM for shared-memory traffic in the product kernel ("Tensor Core operands:
// a matrix instruction still needs a layout contract", fifth paragraph: the
// cost of input conversion belongs in the measurement).
#include <type_traits>

#include "tc_gemm.cuh"

namespace mpg {
namespace {

// Convert 8 consecutive fp32 values into 8 16-bit values (hi) and, for the
// split, 8 lo values (scaled by lo_mul), packed as four 32-bit words each.
__device__ __forceinline__ void convert8(const float (&x)[8], int kind, float scale, float lo_mul, uint4& hi,
                                         uint4& lo) {
  uint32_t w[4], l[4] = {0, 0, 0, 0};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    if (kind == kPassF16) {
      w[j] = pack_f16x2(x[2 * j] * scale, x[2 * j + 1] * scale);   // scale: 1, or 2^s for a split's B
    } else if (kind == kPassBF16) {
      w[j] = pack_bf16x2(x[2 * j] * scale, x[2 * j + 1] * scale);
    } else {
      split_pair(x[2 * j], x[2 * j + 1], scale, lo_mul, w[j], l[j]);
    }
  }
  hi = make_uint4(w[0], w[1], w[2], w[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

struct PassJobs {
  PassJob job[2];
  int64_t items0, total;   // work items of job 0, of both
};

// One work item = 8 consecutive elements of one line of one operand; the
// items of both operands form one index range.  Each thread handles two
// items per loop trip, loading both before converting either.
__global__ void __launch_bounds__(256) prepass_kernel(const __grid_constant__ PassJobs J) {
  griddep_launch_dependents();   // the product may set itself up meanwhile
  const int64_t step = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i0 < J.total; i0 += 2 * step) {
    float x[2][8];
    int64_t o[2];
    int jb[2];
    bool live[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int64_t i = i0 + u * step;
      live[u] = i < J.total;
      jb[u] = (live[u] && i >= J.items0) ? 1 : 0;
      const PassJob& P = J.job[jb[u]];
      const int64_t ii = live[u] ? (jb[u] ? i - J.items0 : i) : 0;
      const int64_t items_per_line = (P.inner + 7) / 8;
      const int64_t per_batch = P.outer * items_per_line;
      const int64_t b = ii / per_batch;
      const int64_t r = ii - b * per_batch;
      const int64_t line = r / items_per_line;
      const int64_t c = (r - line * items_per_line) * 8;
      const float* src = P.in + b * P.stride_in + line * P.ld_in + c;
      o[u] = b * P.outer * P.ld_out + line * P.ld_out + c;   // ld_out % 8 == 0: 16-byte aligned
      if (live[u] && P.vec && c + 7 < P.inner) {
        const float4 v0 = __ldg(reinterpret_cast<const float4*>(src));
        const float4 v1 = __ldg(reinterpret_cast<const float4*>(src) + 1);
        x[u][0] = v0.x; x[u][1] = v0.y; x[u][2] = v0.z; x[u][3] = v0.w;
        x[u][4] = v1.x; x[u][5] = v1.y; x[u][6] = v1.z; x[u][7] = v1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) x[u][e] = (live[u] && c + e < P.inner) ? __ldg(src + e) : 0.0f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (!live[u]) continue;
      const PassJob& P = J.job[jb[u]];
      uint4 h, l;
      convert8(x[u], P.kind, P.scale, P.lo_mul, h, l);
      *reinterpret_cast<uint4*>(P.hi + o[u]) = h;
      if (P.kind == kPassSplit) *reinterpret_cast<uint4*>(P.lo + o[u]) = l;
    }
  }
}

// Copy of a matrix TMA cannot describe (unaligned base, leading dimension or
// batch stride) into a dense layout whose lines start on 16-byte boundaries:
// `batch` matrices of `outer` lines of `inner` elements of ES bytes, read with
// ld_in / stride_in, written with ld_out (a multiple of 8 elements) and
// stride outer * ld_out.  One work item = 8 consecutive elements of a line.
template <int ES>
__global__ void __launch_bounds__(256) copy_pad_kernel(const uint8_t* __restrict__ in, int64_t ld_in,
                                                       int64_t stride_in, int64_t outer, int64_t inner, int64_t batch,
                                                       uint8_t* __restrict__ out, int64_t ld_out) {
  griddep_launch_dependents();   // the product may set itself up meanwhile
  using E = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
  const E* src = reinterpret_cast<const E*>(in);
  E* dst = reinterpret_cast<E*>(out);
  const int64_t items_per_line = (inner + 7) / 8;
  const int64_t per_batch = outer * items_per_line;
  const int64_t total = per_batch * batch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per_batch;
    const int64_t r = i - b * per_batch;
    const int64_t line = r / items_per_line;
    const int64_t c = (r - line * items_per_line) * 8;
    const E* s = src + b * stride_in + line * ld_in + c;
    E v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (c + e < inner) ? __ldg(s + e) : E(0);
    E* d = dst + (b * outer + line) * ld_out + c;   // 16-byte aligned (ld_out % 8 == 0)
    if constexpr (ES == 2) {
      *reinterpret_cast<uint4*>(d) = make_uint4(v[0] | ((uint32_t)v[1] << 16), v[2] | ((uint32_t)v[3] << 16),
                                                v[4] | ((uint32_t)v[5] << 16), v[6] | ((uint32_t)v[7] << 16));
    } else {
      reinterpret_cast<uint4*>(d)[0] = make_uint4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<uint4*>(d)[1] = make_uint4(v[4], v[5], v[6], v[7]);
    }
  }
}

// Transposed copy of 32-bit elements: `batch` matrices of `outer` lines of
// `inner` elements (ld_in, stride_in) become `inner` lines of `outer`
// elements with ld_out (a multiple of 8) and stride inner * ld_out.  32 x 32
// tiles through shared memory (one padding column against bank conflicts),
// both global sides coalesced.
__global__ void __launch_bounds__(256) transpose32_kernel(const uint32_t* __restrict__ in, int64_t ld_in,
                                                          int64_t stride_in, int64_t outer, int64_t inner,
                                                          uint32_t* __restrict__ out, int64_t ld_out) {
  __shared__ uint32_t tile[32][33];
  griddep_launch_dependents();   // the product may set itself up meanwhile
  const int64_t b = blockIdx.z;
  const int64_t o0 = (int64_t)blockIdx.y * 32, i0 = (int64_t)blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;   // 32 x 8 threads
  const uint32_t* src = in + b * stride_in;
  uint32_t* dst = out + b * inner * ld_out;
#pragma unroll
  for (int r = ty; r < 32; r += 8) {
    const int64_t o = o0 + r, i = i0 + tx;
    tile[r][tx] = (o < outer && i < inner) ? __ldg(src + o * ld_in + i) : 0u;
  }
  __syncthreads();
#pragma unroll
  for (int r = ty; r < 32; r += 8) {
    const int64_t i = i0 + r, o = o0 + tx;
    // the padding columns of each output line (outer .. ld_out-1) are zero
    if (i < inner && o < ld_out) dst[i * ld_out + o] = (o < outer) ? tile[tx][r] : 0u;
  }
}

}  // namespace

cudaError_t launch_transpose32(const void* in, int64_t ld_in, int64_t stride_in, int64_t outer, int64_t inner,
                               int64_t batch, void* out, int64_t ld_out, cudaStream_t stream) {
  if (batch > 65535 || (outer + 31) / 32 > 65535) return cudaErrorInvalidValue;
  // blocks along the output lines also cover their padding columns
  const int64_t out_cols = (ld_out > outer) ? ld_out : outer;
  dim3 grid((unsigned)((inner + 31) / 32), (unsigned)((out_cols + 31) / 32), (unsigned)batch);
  transpose32_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint32_t*>(in), ld_in, stride_in, outer, inner,
                                               static_cast<uint32_t*>(out), ld_out);
  return cudaGetLastError();
}

cudaError_t launch_copy_pad(const void* in, int elem_bytes, int64_t ld_in, int64_t stride_in, int64_t outer,
                            int64_t inner, int64_t batch, void* out, int64_t ld_out, int sm_count,
                            cudaStream_t stream) {
  const int64_t total = batch * outer * ((inner + 7) / 8);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  if (blocks < 1) blocks = 1;
  const uint8_t* src = static_cast<const uint8_t*>(in);
  uint8_t* dst = static_cast<uint8_t*>(out);
  if (elem_bytes == 2)
    copy_pad_kernel<2><<<(int)blocks, 256, 0, stream>>>(src, ld_in, stride_in, outer, inner, batch, dst, ld_out);
  else if (elem_bytes == 4)
    copy_pad_kernel<4><<<(int)blocks, 256, 0, stream>>>(src, ld_in, stride_in, outer, inner, batch, dst, ld_out);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_prepass(const PassJob& a, const PassJob* b, int sm_count, cudaStream_t stream) {
  PassJobs J;
  J.job[0] = a;
  J.job[1] = b ? *b : a;
  for (int i = 0; i < (b ? 2 : 1); ++i) {
    PassJob& P = J.job[i];
    if (P.kind != kPassF16 && P.kind != kPassBF16 && P.kind != kPassSplit) return cudaErrorInvalidValue;
    P.vec = reinterpret_cast<uintptr_t>(P.in) % 16 == 0 && P.ld_in % 4 == 0 && (P.batch == 1 || P.stride_in % 4 == 0);
  }
  auto items = [](const PassJob& P) { return P.batch * P.outer * ((P.inner + 7) / 8); };
  J.items0 = items(J.job[0]);
  J.total = J.items0 + (b ? items(J.job[1]) : 0);
  int64_t blocks = (J.total + 511) / 512;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  if (blocks < 1) blocks = 1;
  prepass_kernel<<<(int)blocks, 256, 0, stream>>>(J);
  return cudaGetLastError();
}

}  // namespace mpg
