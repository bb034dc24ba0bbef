// Instantiations of the tensor-core kernel that stages fp32 operands by TMA
// and converts them in shared memory (fp16 / bf16 rounding, hi/lo split).
#include "tc_gemm.cuh"

namespace mpg {

bool tc_lookup_staged(Conv conv, int bn, TcKernel* out) {
#define MPG_STAGED(CV, OPV, BNV)                                                   \
  if (conv == CV && bn == BNV) return tc_fill<TcTraits<Src::kTmaStaged, CV, OPV, SrcT::kF32, BNV>>(out);
  MPG_STAGED(Conv::kRoundF16, Op::kF16, 256)
  MPG_STAGED(Conv::kRoundF16, Op::kF16, 128)
  MPG_STAGED(Conv::kRoundF16, Op::kF16, 64)
  MPG_STAGED(Conv::kRoundBF16, Op::kBF16, 256)
  MPG_STAGED(Conv::kRoundBF16, Op::kBF16, 128)
  MPG_STAGED(Conv::kRoundBF16, Op::kBF16, 64)
  MPG_STAGED(Conv::kSplit3, Op::kF16, 128)
  MPG_STAGED(Conv::kSplit3, Op::kF16, 64)
  MPG_STAGED(Conv::kSplitA2, Op::kF16, 128)
  MPG_STAGED(Conv::kSplitA2, Op::kF16, 64)
  MPG_STAGED(Conv::kSplit4, Op::kF16, 64)
  MPG_STAGED(Conv::kSplit1, Op::kF16, 128)
  MPG_STAGED(Conv::kSplit1, Op::kF16, 64)
  MPG_STAGED(Conv::kSplit3M, Op::kF16, 128)
  MPG_STAGED(Conv::kSplit3M, Op::kF16, 64)
#undef MPG_STAGED
  return false;
}

}  // namespace mpg
