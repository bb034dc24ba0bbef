// Internal structures shared between the host planner (api.cu) and the kernel
// translation units.  Not part of the public C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mpg {

// Where the operands of the tensor-core kernel come from.
enum class Src : int {
  kTmaDirect = 0,  // TMA straight into the MMA operand stages (16-bit or tf32 data)
  kTmaStaged = 1,  // TMA of fp32 into staging buffers, converter warps -> fp16/bf16 stages
  kGeneric = 2,    // converter warps load from global memory (any alignment)
};

// What the converter does to each fp32 (or 16-bit) element.
enum class Conv : int {
  kNone = 0,      // operand used as stored (direct path, or a plain copy)
  kRoundF16 = 1,  // fp32 -> fp16 round-to-nearest-even
  kRoundBF16 = 2, // fp32 -> bf16 round-to-nearest-even
  kSplit3 = 3,    // fp32 -> hi, lo*2^11; three accumulator chains
  kSplit1 = 4,    // fp32 -> hi, lo; one shared accumulator chain
  kSplitA2 = 5,   // A: fp32 -> hi, lo*2^11; B: fp32 -> fp16; two chains (A_hi B, A_lo B)
  kSplit4 = 6,    // fp32 -> hi, lo*2^11; four chains (hh, hl, lh, ll)
  kSplit3M = 7,   // fp32 -> hi, lo*2^L; two accumulators, hh and hl + lh (one K chunk)
};

// Bits of the device status word.
enum : uint32_t {
  kStatusTimeout = 1u << 0,  // some bounded wait expired
  kStatusBadArg = 1u << 1,   // a kernel saw arguments it cannot honour
};

// Element type the tensor core consumes.
enum class Op : int { kF16 = 0, kBF16 = 1, kTF32 = 2 };

// Storage type of the source operand.
enum class SrcT : int { kF32 = 0, kF16 = 1, kBF16 = 2 };

struct TcParams {
  CUtensorMap map_a;  // used by the TMA paths only
  CUtensorMap map_b;
  CUtensorMap map_a_lo;  // direct split path: the lo halves of pre-split operands
  CUtensorMap map_b_lo;
  CUtensorMap map_out;  // fp32 destination of TMA stores: C, or the split-K partials {n, m, splits*batch}
  int32_t tma_store;    // 1: the epilogue stores its 32 x 32 blocks by TMA (fp32, beta == 0, aligned)
  const void* a;      // generic path addressing (element units of the source type)
  const void* b;
  int64_t lda, ldb, stride_a, stride_b;
  void* c;            // output, element type c_dtype
  int64_t ldc, stride_c;
  float* partial;     // split-K partial sums [split][batch][m][n] (ld = n), or null
  int32_t m, n, k, batch;
  int32_t a_mn_major, b_mn_major;  // 1: operand stored with M (resp. N) contiguous
  int32_t num_m_blk, num_n_blk, num_k_blk;
  int32_t splits, kb_per_split;
  int32_t num_tiles;
  int32_t group_m;
  int32_t c_dtype;    // 0 fp32, 1 fp16, 2 bf16 (rounded once, to nearest even, when stored)
  int32_t c_vec_ok;   // 4-element vectors of C are aligned (base, ldc % 4, batch stride % 4)
  int32_t a_vec_ok, b_vec_ok;  // 4-element chunks of A / B are vector-aligned (generic loads)
  int32_t p_vec_ok;   // partial buffer: n % 4 == 0
  float alpha;        // already multiplied by 2^-(split_exp_a + split_exp_b)
  float beta;
  float scale_a, scale_b;  // 2^split_exp_a, 2^split_exp_b (split converter)
  float lo_mul, lo_inv;    // split: the lo half's scale 2^L and its inverse (L = 11 or 0)
  uint32_t* status;
  uint64_t wait_limit_ns;
  int32_t chunk_kb;   // k-blocks per accumulation chunk (0: the whole k range of a tile)
  // split tail (CTA-pair kernel): work items from tail_first on are halves
  // of the k range of the last tiles, cut at k-block tail_kb_mid; each half
  // writes its partial sums to tail_ws and counts itself in tail_cnt (zero
  // at launch); the second half to arrive adds the first's and stores C.
  // tail_first = num_tiles: no split tail.
  int32_t tail_first;
  int32_t tail_kb_mid;
  float* tail_ws;
  uint32_t* tail_cnt;
};

struct LaunchInfo {
  int grid;
  int block;
  int smem_bytes;
};

// One instantiated tensor-core kernel: its launch shape and entry.
struct TcKernel {
  const void* fn;
  int block;
  int smem_bytes;
  int bn;
};

// Look up the tensor-core kernel for a configuration; returns false if this
// combination is not instantiated.
bool tc_kernel_lookup(Src src, Conv conv, Op op, SrcT st, int bn, TcKernel* out);

// Copy into a dense layout with 16-byte aligned lines (ld_out % 8 == 0);
// elem_bytes 2 or 4.
cudaError_t launch_copy_pad(const void* in, int elem_bytes, int64_t ld_in, int64_t stride_in, int64_t outer,
                            int64_t inner, int64_t batch, void* out, int64_t ld_out, int sm_count,
                            cudaStream_t stream);

// Transposed copy of 32-bit elements: `outer` lines of `inner` become `inner`
// lines of `outer` (ld_out % 8 == 0, padding columns zeroed).
cudaError_t launch_transpose32(const void* in, int64_t ld_in, int64_t stride_in, int64_t outer, int64_t inner,
                               int64_t batch, void* out, int64_t ld_out, cudaStream_t stream);

// Fused prompt attention O = softmax(scale * Q K^T) V (head dimension 128).
// Keys per block of the fused attention (the K and V tensor maps' box).
constexpr int kAttnKeyBlock = 128;

struct AttnParams {
  CUtensorMap map_k;   // K: fp16 [lk][ldk], box 64 dims x kAttnKeyBlock keys
  CUtensorMap map_v;   // V: fp16 [lk][ldv], box 64 dims x kAttnKeyBlock / 2 keys
  const float* q;      // fp32 [lq][ldq]
  int64_t ldq;
  float* o;            // fp32 [lq][ldo]
  int64_t ldo;
  float* part_o;       // key splits > 1: unnormalised partial outputs [split][lq][128]
  float* part_m;       //   and their row maxima [split][lq] (log2 domain)
  float* part_l;       //   and row sums [split][lq]
  int32_t lq, lk;
  int32_t splits, kb_per_split, num_q_blk;
  int32_t q_vec_ok;    // Q rows are 16-byte aligned (float4 loads)
  float scale_log2;    // softmax scale * log2(e)
  uint32_t* status;
  uint64_t wait_limit_ns;
};
cudaError_t launch_attention(const AttnParams& p, bool two_chain, cudaStream_t stream);
int attention_smem_bytes();

// The 16-bit and tf32 direct product on a CTA pair (cta_group::2, 256 x 256
// tiles per cluster of two CTAs), and the three-chain split on the
// conversion pass's fp16 copies (256 x 128 tiles); false for combinations it
// does not cover.
bool tc_lookup_pair(Op op, Conv conv, TcKernel* out);

// Plain fp32 FFMA comparator.
struct FfmaParams {
  const float* a;
  const float* b;
  void* c;
  int32_t c_dtype;
  int64_t lda, ldb, ldc, stride_a, stride_b, stride_c;
  int32_t m, n, k, batch;
  int32_t a_col_major, b_col_major;
  float alpha, beta;
};
cudaError_t launch_ffma(const FfmaParams& p, cudaStream_t stream);

// C = beta * C (beta == 0: C = 0 without reading it).
cudaError_t launch_scale_c(void* c, int c_dtype, int64_t ldc, int64_t stride_c, int32_t m, int32_t n,
                           int32_t batch, float beta, cudaStream_t stream);

// C = alpha * sum_s partial[s] + beta * C, partial laid out [split][batch][m][n].
cudaError_t launch_splitk_reduce(const float* partial, int32_t splits, void* c, int c_dtype, int64_t ldc,
                                 int64_t stride_c, int32_t m, int32_t n, int32_t batch, float alpha, float beta,
                                 cudaStream_t stream);

cudaError_t launch_probe_mma(const void* a, const void* b, float* d, cudaStream_t stream);

// Separate conversion pass: a stored fp32 matrix (per batch `outer` lines of
// `inner` elements, leading dimension ld_in, batch stride stride_in) into
// packed 16-bit copies with leading dimension ld_out (batch stride
// outer * ld_out).  kind: fp16 or bf16 rounding of x*scale, or the split
// hi = fp16(x*scale), lo = fp16((x*scale - hi) * lo_mul) (lo written for
// the split only).  scale and lo_mul are powers of two.  One launch converts
// one or two operands.
enum : int { kPassF16 = 0, kPassBF16 = 1, kPassSplit = 2 };
struct PassJob {
  const float* in;
  int64_t ld_in, stride_in, outer, inner, batch;
  uint16_t* hi;
  uint16_t* lo;
  int64_t ld_out;
  float scale, lo_mul;
  int kind;
  int vec;   // set by the launcher
};
cudaError_t launch_prepass(const PassJob& a, const PassJob* b, int sm_count, cudaStream_t stream);
cudaError_t launch_probe_mma_frag(const uint32_t* a, const uint32_t* b, float* d, cudaStream_t stream);
cudaError_t launch_probe_staging(const float* in, float* out, int64_t blocks, int scalar, int sm_count,
                                 cudaStream_t stream);
cudaError_t launch_selftest_wait(uint32_t* status, uint64_t limit_ns, cudaStream_t stream);
// fp32 multiply-add throughput: `blocks` blocks of 256 threads, each thread
// 32 x iters independent fmaf (scalar or packed pairs).
cudaError_t launch_probe_fma(float* out, int64_t blocks, int iters, int packed, cudaStream_t stream);
// One-CTA tcgen05 pass (M 128, N n, K 64) whose TMEM accumulator is copied
// out unscattered, register by register (n = 64, 128 or 256).
cudaError_t launch_probe_tmem(const void* a, const void* b, int n, float* d, uint32_t* status, uint64_t limit_ns,
                              cudaStream_t stream);
// The same on a cluster of two CTAs (cta_group::2, M = 256): A 256 x 64,
// the CTA of rank r holding rows 128r .. 128r+127; B n x 64 split between
// the CTAs by columns.
cudaError_t launch_probe_tmem_pair(const void* a, const void* b, int n, float* d, uint32_t* status,
                                   uint64_t limit_ns, cudaStream_t stream);

// Device status word of the current device (allocated by the runtime as a
// module global; one per device).
uint32_t* status_word_ptr();

}  // namespace mpg
