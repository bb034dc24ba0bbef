// Instantiations of the tensor-core kernel whose converter warps read the
// operands with plain global loads: any alignment and any leading dimension
// (the path for layouts TMA cannot describe).
#include "tc_gemm.cuh"

namespace mpg {

bool tc_lookup_generic(Conv conv, Op op, SrcT st, int bn, TcKernel* out) {
#define MPG_GENERIC(CV, OPV, STV, BNV)                                                         \
  if (conv == CV && op == OPV && st == STV && bn == BNV)                                       \
    return tc_fill<TcTraits<Src::kGeneric, CV, OPV, STV, BNV>>(out);
  MPG_GENERIC(Conv::kNone, Op::kF16, SrcT::kF16, 128)
  MPG_GENERIC(Conv::kNone, Op::kBF16, SrcT::kBF16, 128)
  MPG_GENERIC(Conv::kNone, Op::kTF32, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kRoundF16, Op::kF16, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kRoundBF16, Op::kBF16, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kSplit3, Op::kF16, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kSplit1, Op::kF16, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kSplitA2, Op::kF16, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kSplit4, Op::kF16, SrcT::kF32, 64)
  // 64-wide tiles for products with fewer tiles than SMs
  MPG_GENERIC(Conv::kNone, Op::kF16, SrcT::kF16, 64)
  MPG_GENERIC(Conv::kNone, Op::kBF16, SrcT::kBF16, 64)
  MPG_GENERIC(Conv::kNone, Op::kTF32, SrcT::kF32, 64)
  MPG_GENERIC(Conv::kRoundF16, Op::kF16, SrcT::kF32, 64)
  MPG_GENERIC(Conv::kRoundBF16, Op::kBF16, SrcT::kF32, 64)
  MPG_GENERIC(Conv::kSplit3, Op::kF16, SrcT::kF32, 64)
  MPG_GENERIC(Conv::kSplit1, Op::kF16, SrcT::kF32, 64)
  MPG_GENERIC(Conv::kSplitA2, Op::kF16, SrcT::kF32, 64)
  MPG_GENERIC(Conv::kSplit3M, Op::kF16, SrcT::kF32, 128)
  MPG_GENERIC(Conv::kSplit3M, Op::kF16, SrcT::kF32, 64)
#undef MPG_GENERIC
  return false;
}

}  // namespace mpg
