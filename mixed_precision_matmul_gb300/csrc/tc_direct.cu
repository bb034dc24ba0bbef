// Instantiations of the tensor-core kernel whose operands arrive by TMA
// straight into the MMA stages (fp16 / bf16 via kind::f16, fp32 via kind::tf32,
// and fp16 hi/lo halves written by the separate conversion pass).
#include "tc_gemm.cuh"

namespace mpg {

bool tc_lookup_direct(Conv conv, Op op, int bn, TcKernel* out) {
  // pre-split fp16 operands (hi and lo halves loaded by TMA)
#define MPG_DIRECT_SPLIT(CV, BNV)                                                   \
  if (conv == CV && bn == BNV) return tc_fill<TcTraits<Src::kTmaDirect, CV, Op::kF16, SrcT::kF16, BNV>>(out);
  MPG_DIRECT_SPLIT(Conv::kSplit3, 128)
  MPG_DIRECT_SPLIT(Conv::kSplit3, 64)
  MPG_DIRECT_SPLIT(Conv::kSplit1, 128)
  MPG_DIRECT_SPLIT(Conv::kSplit1, 64)
  MPG_DIRECT_SPLIT(Conv::kSplitA2, 128)
  MPG_DIRECT_SPLIT(Conv::kSplitA2, 64)
  MPG_DIRECT_SPLIT(Conv::kSplit4, 64)
  MPG_DIRECT_SPLIT(Conv::kSplit3M, 128)
  MPG_DIRECT_SPLIT(Conv::kSplit3M, 64)
#undef MPG_DIRECT_SPLIT
  if (conv != Conv::kNone) return false;
#define MPG_DIRECT(OPV, STV, BNV)                                                  \
  if (op == OPV && bn == BNV) return tc_fill<TcTraits<Src::kTmaDirect, Conv::kNone, OPV, STV, BNV>>(out);
  MPG_DIRECT(Op::kF16, SrcT::kF16, 256)
  MPG_DIRECT(Op::kF16, SrcT::kF16, 128)
  MPG_DIRECT(Op::kF16, SrcT::kF16, 64)
  MPG_DIRECT(Op::kBF16, SrcT::kBF16, 256)
  MPG_DIRECT(Op::kBF16, SrcT::kBF16, 128)
  MPG_DIRECT(Op::kBF16, SrcT::kBF16, 64)
  MPG_DIRECT(Op::kTF32, SrcT::kF32, 256)
  MPG_DIRECT(Op::kTF32, SrcT::kF32, 128)
  MPG_DIRECT(Op::kTF32, SrcT::kF32, 64)
#undef MPG_DIRECT
  return false;
}

}  // namespace mpg
