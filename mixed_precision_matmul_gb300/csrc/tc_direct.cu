// Instantiations of the tensor-core kernel whose operands arrive by TMA
// straight into the MMA stages (fp16 / bf16 via kind::f16, fp32 via kind::tf32).
#include "tc_gemm.cuh"

namespace mpg {

bool tc_lookup_direct(Op op, int bn, TcKernel* out) {
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
