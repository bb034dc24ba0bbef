// Separate conversion pass of the fp32 operands: fp32 -> fp16 / bf16
// (round to nearest even) or the fp16 hi/lo split, written as packed 16-bit
// copies that the direct TMA path then multiplies.  The arithmetic is the
// converter warps' (same conversions, same split), so both routes give the
// same operands; this one trades one extra read and write of the operands in
// HBM for shared-memory traffic in the product kernel ("Tensor Core operands:
// a matrix instruction still needs a layout contract", fifth paragraph: the
// cost of input conversion belongs in the measurement).
#include "tc_gemm.cuh"

namespace mpg {
namespace {

template <Conv CV>
__global__ void __launch_bounds__(256) prepass_kernel(const float* __restrict__ in, int64_t ld_in,
                                                      int64_t stride_in, int64_t outer, int64_t inner,
                                                      int64_t batch, uint16_t* __restrict__ hi,
                                                      uint16_t* __restrict__ lo, int64_t ld_out, float scale,
                                                      int vec) {
  const int64_t chunks_per_line = (inner + 3) / 4;
  const int64_t per_batch = outer * chunks_per_line;
  const int64_t total = per_batch * batch;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / per_batch;
    const int64_t r = i - b * per_batch;
    const int64_t line = r / chunks_per_line;
    const int64_t c = (r - line * chunks_per_line) * 4;
    const float* src = in + b * stride_in + line * ld_in + c;
    float x[4];
    if (vec && c + 3 < inner) {
      const float4 v = __ldg(reinterpret_cast<const float4*>(src));
      x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) x[e] = (c + e < inner) ? __ldg(src + e) : 0.0f;
    }
    uint32_t w0, w1, l0 = 0, l1 = 0;
    if constexpr (CV == Conv::kRoundF16) {
      w0 = pack_f16x2(x[0], x[1]);
      w1 = pack_f16x2(x[2], x[3]);
    } else if constexpr (CV == Conv::kRoundBF16) {
      w0 = pack_bf16x2(x[0], x[1]);
      w1 = pack_bf16x2(x[2], x[3]);
    } else {
      constexpr int L = (CV == Conv::kSplit3) ? 11 : 0;
      split_pair<L>(x[0], x[1], scale, w0, l0);
      split_pair<L>(x[2], x[3], scale, w1, l1);
    }
    const int64_t o = b * outer * ld_out + line * ld_out + c;   // ld_out % 8 == 0: 8-byte aligned
    *reinterpret_cast<uint2*>(hi + o) = make_uint2(w0, w1);
    if constexpr (CV == Conv::kSplit3 || CV == Conv::kSplit1) *reinterpret_cast<uint2*>(lo + o) = make_uint2(l0, l1);
  }
}

}  // namespace

cudaError_t launch_prepass(Conv conv, const float* in, int64_t ld_in, int64_t stride_in, int64_t outer,
                           int64_t inner, int64_t batch, uint16_t* hi, uint16_t* lo, int64_t ld_out, float scale,
                           int sm_count, cudaStream_t stream) {
  const int64_t total = batch * outer * ((inner + 3) / 4);
  int64_t blocks = (total + 255) / 256;
  if (blocks > (int64_t)sm_count * 16) blocks = (int64_t)sm_count * 16;
  if (blocks < 1) blocks = 1;
  const int vec = reinterpret_cast<uintptr_t>(in) % 16 == 0 && ld_in % 4 == 0 && (batch == 1 || stride_in % 4 == 0);
  switch (conv) {
    case Conv::kRoundF16:
      prepass_kernel<Conv::kRoundF16><<<(int)blocks, 256, 0, stream>>>(in, ld_in, stride_in, outer, inner, batch, hi,
                                                                        lo, ld_out, scale, vec);
      break;
    case Conv::kRoundBF16:
      prepass_kernel<Conv::kRoundBF16><<<(int)blocks, 256, 0, stream>>>(in, ld_in, stride_in, outer, inner, batch,
                                                                         hi, lo, ld_out, scale, vec);
      break;
    case Conv::kSplit3:
      prepass_kernel<Conv::kSplit3><<<(int)blocks, 256, 0, stream>>>(in, ld_in, stride_in, outer, inner, batch, hi, lo,
                                                                      ld_out, scale, vec);
      break;
    case Conv::kSplit1:
      prepass_kernel<Conv::kSplit1><<<(int)blocks, 256, 0, stream>>>(in, ld_in, stride_in, outer, inner, batch, hi, lo,
                                                                      ld_out, scale, vec);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace mpg
