// The product's C entry points (include/mpgemm.h): options, workspace
// queries, mpg_gemm / mpg_gemm_ex, the allocation-free form, the device
// status word, the probes and the bounded-wait self test.  Nothing here
// allocates device memory.
#include <cmath>
#include <cstring>

#include "host.h"

using namespace mpg;

namespace {

// Scratch of mpg_gemm_noalloc: split-K partial sums for callers that cannot
// allocate.  A module global, so every device that loads the library holds
// one copy.  In host code this name is only a stand-in for the symbol, never
// a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[MPG_NOALLOC_SCRATCH_BYTES / sizeof(float)];

struct NoallocSlot {
  bool ready = false;
  void* ptr = nullptr;
};
NoallocSlot g_noalloc[kMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
mpg_status noalloc_scratch(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(MPG_ERR_NO_DEVICE, "no current CUDA device");
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocSlot& slot = g_noalloc[dev];
  if (!slot.ready) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
      cudaGetLastError();
      return fail(MPG_ERR_CUDA, "cannot resolve the static scratch on device %d: %s", dev, cudaGetErrorString(e));
    }
    slot.ptr = ptr;
    slot.ready = true;
  }
  *out = slot.ptr;
  return MPG_OK;
}

}  // namespace

extern "C" {

void mpg_options_init(mpg_options* opt) {
  if (!opt) return;
  std::memset(opt, 0, sizeof(*opt));
}

int mpg_version(void) { return 100; }

const char* mpg_last_error_string(void) { return t_err.c_str(); }

namespace {
// Workspace of everything but the split tail, from the sizes alone.  With
// copy_room, large 16-bit and tf32 products also get room for aligned
// copies of both operands (the sizes-only query cannot see whether the
// operands need them).
size_t regions_bytes(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_precision mode, const mpg_options* opt,
                     bool copy_room) {
  mpg_options o;
  resolve_options(opt, &o);
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0 || mode == MPG_FP32_FFMA) return 0;
  DeviceInfo* dev = nullptr;
  int sm = 152;
  if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
  t_err.clear();
  const size_t partials = splitk_bytes(choose_splits(m, n, k, batch, sm, o), m, n, batch);
  if (copy_room && !o.force_generic_load && o.prepass >= 0 && (mode == MPG_FP16_F32ACC || mode == MPG_BF16_F32ACC ||
                                                  mode == MPG_TF32) &&
      auto_prepass_shape(m, n, k)) {
    // Large 16-bit and tf32 products: room for copies of both operands with
    // 16-byte aligned lines, in whichever majorness the direct path needs,
    // so that operands TMA cannot describe as given (unaligned base,
    // leading dimension or batch stride; tf32 in the wrong majorness) are
    // copied and multiplied on the TMA path rather than loaded element by
    // element.  The same room holds the conversion pass's 16-bit copies of
    // fp32 operands in the fp16 / bf16 modes.  2 bytes per element (4 for
    // tf32) at the worse of the two line paddings.
    const size_t es = (mode == MPG_TF32) ? 4 : 2;
    auto pad8 = [](int64_t x) { return (x + 7) / 8 * 8; };
    const size_t a = align256((size_t)batch * (size_t)std::max(m * pad8(k), k * pad8(m)) * es);
    const size_t b = align256((size_t)batch * (size_t)std::max(k * pad8(n), n * pad8(k)) * es);
    return align256(partials) + a + b;
  }
  if ((o.prepass == 1 && prepass_mode(mode)) ||
      (o.prepass == 0 && split_mode(mode) && auto_prepass_shape(m, n, k))) {
    // layouts are not known here: take the larger of the two line paddings
    const bool split_b =
        (mode == MPG_SPLIT_FP16_3CHAIN || mode == MPG_SPLIT_FP16_1CHAIN || mode == MPG_SPLIT_FP16_4CHAIN);
    const bool split_a = split_b || mode == MPG_SPLIT_A_FP16_2CHAIN;
    size_t worst = 0;
    for (mpg_layout al : {MPG_ROW_MAJOR, MPG_COL_MAJOR})
      for (mpg_layout bl : {MPG_ROW_MAJOR, MPG_COL_MAJOR})
        worst = std::max(worst, prepass_layout(m, n, k, batch, al, bl, split_a, split_b, partials).end);
    return worst;
  }
  return partials;
}

// Split-tail bound for these sizes (0 when it cannot apply).
size_t tail_region(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_precision mode, const mpg_options* opt) {
  mpg_options o;
  resolve_options(opt, &o);
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0) return 0;
  DeviceInfo* dev = nullptr;
  int sm = 152;
  if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
  t_err.clear();
  return tail_bound(m, n, k, batch, mode, sm, o);
}
}  // namespace

size_t mpg_gemm_workspace_size(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_precision mode,
                               const mpg_options* opt) {
  const size_t r = regions_bytes(m, n, k, batch, mode, opt, true);
  const size_t t = tail_region(m, n, k, batch, mode, opt);
  return t ? align256(r) + t : r;
}

size_t mpg_gemm_workspace_size_ex(int64_t m, int64_t n, int64_t k, int64_t batch, const void* A, int64_t lda,
                                  int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout, const void* B,
                                  int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                                  mpg_precision mode, const mpg_options* opt) {
  mpg_options o;
  resolve_options(opt, &o);
  const size_t base = regions_bytes(m, n, k, batch, mode, opt, false);
  const size_t tail = tail_region(m, n, k, batch, mode, opt);
  auto with_tail = [&](size_t r) { return tail ? align256(r) + tail : r; };
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0 || o.force_generic_load) return with_tail(base);
  // the aligned copies the planner makes for 16-bit (or tf32 K-major)
  // operands on the direct path that TMA cannot describe as given
  const bool f16in = (mode == MPG_FP16_F32ACC && a_dtype == MPG_F16 && b_dtype == MPG_F16) ||
                     (mode == MPG_BF16_F32ACC && a_dtype == MPG_BF16 && b_dtype == MPG_BF16);
  const bool tf32 = (mode == MPG_TF32 && a_dtype == MPG_F32 && b_dtype == MPG_F32);
  // fp16 / bf16 modes on fp32 operands: the conversion pass on large products
  const bool round_f32 = (mode == MPG_FP16_F32ACC || mode == MPG_BF16_F32ACC) && a_dtype == MPG_F32 &&
                         b_dtype == MPG_F32;
  if (round_f32 && o.prepass == 0 && auto_prepass_shape(m, n, k)) {
    DeviceInfo* dev = nullptr;
    int sm = 152;
    if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
    t_err.clear();
    const PrepassLayout L = prepass_layout(m, n, k, batch, a_layout, b_layout, false, false,
                                           splitk_bytes(choose_splits(m, n, k, batch, sm, o), m, n, batch));
    return with_tail(std::max(base, L.end));
  }
  if (!f16in && !tf32) return with_tail(base);
  Operand Aop{A, lda, strideA, a_dtype, a_layout};
  Operand Bop{B, ldb, strideB, b_dtype, b_layout};
  const mpg_layout a_out = tf32 ? MPG_ROW_MAJOR : a_layout, b_out = tf32 ? MPG_COL_MAJOR : b_layout;
  const bool ca = !tma_ok(Aop, batch) || a_layout != a_out, cb = !tma_ok(Bop, batch) || b_layout != b_out;
  if (!ca && !cb) return with_tail(base);
  DeviceInfo* dev = nullptr;
  int sm = 152;
  if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
  t_err.clear();
  const CopyLayout L = copy_layout(m, n, k, batch, Aop, Bop, ca, cb,
                                   splitk_bytes(choose_splits(m, n, k, batch, sm, o), m, n, batch), a_out, b_out);
  return with_tail(std::max(base, L.end));
}

mpg_status mpg_gemm_ex(int64_t m, int64_t n, int64_t k, int64_t batch, const void* A, int64_t lda,
                       int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout, const void* B, int64_t ldb,
                       int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout, float* C, int64_t ldc,
                       int64_t strideC, float alpha, float beta, mpg_precision mode, void* workspace,
                       size_t workspace_bytes, void* stream, const mpg_options* opt) {
  t_err.clear();
  mpg_options o;
  resolve_options(opt, &o);
  Operand Aop{A, lda, strideA, a_dtype, a_layout};
  Operand Bop{B, ldb, strideB, b_dtype, b_layout};
  mpg_status s = validate(m, n, k, batch, Aop, Bop, C, ldc, strideC, alpha, mode, o);
  if (s != MPG_OK) return s;
  if (m == 0 || n == 0 || batch == 0) return MPG_OK;
  if (workspace && reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
    return fail(MPG_ERR_INVALID_ARG, "workspace not 16-byte aligned");
  if (!workspace) workspace_bytes = 0;
  DeviceInfo* dev = nullptr;
  s = get_device(&dev);
  if (s != MPG_OK) return s;
  Plan plan;
  s = make_plan(m, n, k, batch, Aop, Bop, alpha, mode, o, dev->sm_count, workspace_bytes, &plan);
  if (s != MPG_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t sc = strideC ? strideC : m * ldc;
  cudaError_t e = cudaSuccess;
  switch (plan.kind) {
    case Kind::kNoop:
      return MPG_OK;
    case Kind::kScale:
      e = launch_scale_c(C, o.c_dtype, ldc, sc, (int32_t)m, (int32_t)n, (int32_t)batch, beta, st);
      break;
    case Kind::kFfma: {
      FfmaParams fp;
      fp.a = static_cast<const float*>(A);
      fp.b = static_cast<const float*>(B);
      fp.c = C;
      fp.c_dtype = o.c_dtype;
      fp.lda = lda;
      fp.ldb = ldb;
      fp.ldc = ldc;
      fp.a_col_major = (a_layout == MPG_COL_MAJOR);
      fp.b_col_major = (b_layout == MPG_COL_MAJOR);
      fp.stride_a = strideA ? strideA : (fp.a_col_major ? k * lda : m * lda);
      fp.stride_b = strideB ? strideB : (fp.b_col_major ? n * ldb : k * ldb);
      fp.stride_c = sc;
      fp.m = (int32_t)m;
      fp.n = (int32_t)n;
      fp.k = (int32_t)k;
      fp.batch = (int32_t)batch;
      fp.alpha = alpha;
      fp.beta = beta;
      e = launch_ffma(fp, st);
      break;
    }
    case Kind::kTc: {
      if (plan.copy_a || plan.copy_b) {
        // aligned copies in the workspace, then the direct path on them
        const bool tf32 = (plan.op == Op::kTF32);
        const CopyLayout L = copy_layout(m, n, k, batch, Aop, Bop, plan.copy_a, plan.copy_b,
                                         splitk_bytes(plan.splits, m, n, batch),
                                         tf32 ? MPG_ROW_MAJOR : a_layout, tf32 ? MPG_COL_MAJOR : b_layout);
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        Operand Ac = Aop, Bc = Bop;
        // one copy: same layout (aligned lines) or transposed (32-bit elements)
        auto copy = [&](const void* src, mpg_dtype dt, mpg_layout src_layout, int64_t ld, int64_t stride,
                        mpg_layout dst_layout, int64_t dst_outer, int64_t dst_inner, int64_t dst_ld,
                        uint8_t* dst) -> cudaError_t {
          const int64_t src_outer = (src_layout == dst_layout) ? dst_outer : dst_inner;
          const int64_t s = stride ? stride : src_outer * ld;
          if (src_layout == dst_layout)
            return launch_copy_pad(src, elem_bytes(dt), ld, s, dst_outer, dst_inner, batch, dst, dst_ld,
                                   dev->sm_count, st);
          return launch_transpose32(src, ld, s, dst_inner, dst_outer, batch, dst, dst_ld, st);
        };
        if (plan.copy_a) {
          e = copy(A, a_dtype, a_layout, lda, strideA, L.a_layout, L.a_outer, L.a_inner, L.a_ld, ws + L.off_a);
          Ac = Operand{ws + L.off_a, L.a_ld, L.a_outer * L.a_ld, a_dtype, L.a_layout};
        }
        if (e == cudaSuccess && plan.copy_b) {
          e = copy(B, b_dtype, b_layout, ldb, strideB, L.b_layout, L.b_outer, L.b_inner, L.b_ld, ws + L.off_b);
          Bc = Operand{ws + L.off_b, L.b_ld, L.b_outer * L.b_ld, b_dtype, L.b_layout};
        }
        if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "aligned copy launch: %s", cudaGetErrorString(e));
        return launch_tc(plan, dev, m, n, k, batch, Ac, Bc, C, ldc, strideC, alpha, beta, o, workspace, st, nullptr,
                         nullptr, true);
      }
      if (!plan.prepass)
        return launch_tc(plan, dev, m, n, k, batch, Aop, Bop, C, ldc, strideC, alpha, beta, o, workspace, st);
      // separate conversion pass into the workspace, then the direct path
      const bool sa_ = splits_a(plan.conv), sb_ = splits_b(plan.conv);
      const PrepassLayout L = prepass_layout(m, n, k, batch, a_layout, b_layout, sa_, sb_,
                                             splitk_bytes(plan.splits, m, n, batch));
      uint8_t* ws = static_cast<uint8_t*>(workspace);
      uint16_t* a_hi = reinterpret_cast<uint16_t*>(ws + L.off_a_hi);
      uint16_t* a_lo = sa_ ? reinterpret_cast<uint16_t*>(ws + L.off_a_lo) : nullptr;
      uint16_t* b_hi = reinterpret_cast<uint16_t*>(ws + L.off_b_hi);
      uint16_t* b_lo = sb_ ? reinterpret_cast<uint16_t*>(ws + L.off_b_lo) : nullptr;
      const int ea = sa_ ? o.split_exp_a : 0, eb = sa_ ? o.split_exp_b : 0;
      // the two-chain split splits A only; its B is rounded to fp16
      // the four-chain split uses the three-chain split's halves
      // the two-accumulator split uses the three-chain split's halves too
      const bool three_halves = plan.pre_conv == Conv::kSplitA2 || plan.pre_conv == Conv::kSplit4 ||
                                plan.pre_conv == Conv::kSplit3M;
      const Conv conv_a = three_halves ? Conv::kSplit3 : plan.pre_conv;
      const Conv conv_b = (plan.pre_conv == Conv::kSplitA2) ? Conv::kRoundF16
                          : three_halves                    ? Conv::kSplit3
                                                            : plan.pre_conv;
      const int64_t sA = strideA ? strideA : L.a_outer * lda;
      const int64_t sB = strideB ? strideB : L.b_outer * ldb;
      const float lo_mul = std::ldexp(1.0f, split_lo_exp(plan.pre_conv, o));
      auto kind = [](Conv c) {
        return c == Conv::kRoundF16 ? kPassF16 : c == Conv::kRoundBF16 ? kPassBF16 : kPassSplit;
      };
      // both operands in one launch
      const PassJob ja{static_cast<const float*>(A), lda, sA, L.a_outer, L.a_inner, batch, a_hi, a_lo, L.a_ld,
                       std::ldexp(1.0f, ea), lo_mul, kind(conv_a), 0};
      const PassJob jb{static_cast<const float*>(B), ldb, sB, L.b_outer, L.b_inner, batch, b_hi, b_lo, L.b_ld,
                       std::ldexp(1.0f, eb), lo_mul, kind(conv_b), 0};
      e = launch_prepass(ja, &jb, dev->sm_count, st);
      if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "conversion pass launch: %s", cudaGetErrorString(e));
      const mpg_dtype cdt = (plan.op == Op::kBF16) ? MPG_BF16 : MPG_F16;
      Operand Ah{a_hi, L.a_ld, L.a_outer * L.a_ld, cdt, a_layout};
      Operand Bh{b_hi, L.b_ld, L.b_outer * L.b_ld, cdt, b_layout};
      Operand Al{a_lo, L.a_ld, L.a_outer * L.a_ld, cdt, a_layout};
      Operand Bl{b_lo, L.b_ld, L.b_outer * L.b_ld, cdt, b_layout};
      return launch_tc(plan, dev, m, n, k, batch, Ah, Bh, C, ldc, strideC, alpha, beta, o, workspace, st,
                       sa_ ? &Al : nullptr, sb_ ? &Bl : nullptr, true);
    }
  }
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_gemm(int64_t m, int64_t n, int64_t k, int64_t batch, const void* A, int64_t lda, int64_t strideA,
                    mpg_dtype a_dtype, mpg_layout a_layout, const void* B, int64_t ldb, int64_t strideB,
                    mpg_dtype b_dtype, mpg_layout b_layout, float* C, int64_t ldc, int64_t strideC, float alpha,
                    float beta, mpg_precision mode, void* workspace, size_t workspace_bytes, void* stream) {
  return mpg_gemm_ex(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype, b_layout, C,
                     ldc, strideC, alpha, beta, mode, workspace, workspace_bytes, stream, nullptr);
}

mpg_status mpg_device_status(void* stream) {
  t_err.clear();
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "stream error: %s", cudaGetErrorString(e));
  uint32_t word = 0;
  e = cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  if (word != 0) {
    const uint32_t zero = 0;
    cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice);
    if (word & kStatusTimeout) return fail(MPG_ERR_TIMEOUT, "a kernel gave up a bounded wait (status 0x%x)", word);
    return fail(MPG_ERR_CUDA, "device status 0x%x", word);
  }
  return MPG_OK;
}

mpg_status mpg_probe_mma_m16n8k16(const void* A, const void* B, float* D, void* stream) {
  t_err.clear();
  if (!A || !B || !D) return fail(MPG_ERR_INVALID_ARG, "NULL pointer");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e = launch_probe_mma(A, B, D, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_probe_mma_m16n8k16_fragments(const uint32_t* Afrag, const uint32_t* Bfrag, float* D, void* stream) {
  t_err.clear();
  if (!Afrag || !Bfrag || !D) return fail(MPG_ERR_INVALID_ARG, "NULL pointer");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e = launch_probe_mma_frag(Afrag, Bfrag, D, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_probe_epilogue_staging(const float* in, float* out, int64_t blocks, int scalar, void* stream) {
  t_err.clear();
  if (blocks < 0 || blocks > ((int64_t)1 << 40)) return fail(MPG_ERR_INVALID_ARG, "blocks outside [0, 2^40]");
  if (blocks == 0) return MPG_OK;
  if (!in || !out) return fail(MPG_ERR_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(in) % 16 != 0 || reinterpret_cast<uintptr_t>(out) % 16 != 0)
    return fail(MPG_ERR_INVALID_ARG, "in and out must be 16-byte aligned");
  if (scalar != 0 && scalar != 1) return fail(MPG_ERR_INVALID_ARG, "scalar must be 0 or 1");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e = launch_probe_staging(in, out, blocks, scalar, dev->sm_count, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_probe_fma_rate(float* out, int64_t blocks, int iters, int packed, void* stream) {
  t_err.clear();
  if (!out) return fail(MPG_ERR_INVALID_ARG, "NULL pointer");
  if (reinterpret_cast<uintptr_t>(out) % 4 != 0) return fail(MPG_ERR_INVALID_ARG, "out not aligned to 4 bytes");
  if (blocks < 1 || blocks > 65535) return fail(MPG_ERR_INVALID_ARG, "blocks outside [1, 65535]");
  if (iters < 1 || iters > (1 << 19)) return fail(MPG_ERR_INVALID_ARG, "iters outside [1, 2^19]");
  if (packed != 0 && packed != 1) return fail(MPG_ERR_INVALID_ARG, "packed must be 0 or 1");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e = launch_probe_fma(out, blocks, iters, packed, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_probe_tmem_acc(const void* A, const void* B, int n, float* D, void* stream) {
  t_err.clear();
  if (!A || !B || !D) return fail(MPG_ERR_INVALID_ARG, "NULL pointer");
  if (n != 64 && n != 128 && n != 256) return fail(MPG_ERR_INVALID_ARG, "n must be 64, 128 or 256");
  if (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0)
    return fail(MPG_ERR_INVALID_ARG, "A and B must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(D) % 4 != 0) return fail(MPG_ERR_INVALID_ARG, "D not aligned to 4 bytes");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e = launch_probe_tmem(A, B, n, D, dev->status, 1000000000ull, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_probe_tmem_acc_pair(const void* A, const void* B, int n, float* D, void* stream) {
  t_err.clear();
  if (!A || !B || !D) return fail(MPG_ERR_INVALID_ARG, "NULL pointer");
  if (n != 64 && n != 128 && n != 256) return fail(MPG_ERR_INVALID_ARG, "n must be 64, 128 or 256");
  if (reinterpret_cast<uintptr_t>(A) % 16 != 0 || reinterpret_cast<uintptr_t>(B) % 16 != 0)
    return fail(MPG_ERR_INVALID_ARG, "A and B must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(D) % 4 != 0) return fail(MPG_ERR_INVALID_ARG, "D not aligned to 4 bytes");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaError_t e =
      launch_probe_tmem_pair(A, B, n, D, dev->status, 1000000000ull, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "probe launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

mpg_status mpg_selftest_wait_timeout(int64_t timeout_ns, void* stream) {
  t_err.clear();
  if (timeout_ns < 1000000 || timeout_ns > 10000000000ll)
    return fail(MPG_ERR_INVALID_ARG, "timeout_ns outside [1 ms, 10 s]");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_selftest_wait(dev->status, (uint64_t)timeout_ns, st);
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "self-test launch: %s", cudaGetErrorString(e));
  return mpg_device_status(stream);
}

mpg_status mpg_gemm_noalloc(int64_t m, int64_t n, int64_t k, int64_t batch, const void* A, int64_t lda,
                            int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout, const void* B, int64_t ldb,
                            int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout, float* C, int64_t ldc,
                            int64_t strideC, float alpha, float beta, mpg_precision mode, void* stream,
                            const mpg_options* opt) {
  t_err.clear();
  mpg_options o;
  resolve_options(opt, &o);
  Operand Aop{A, lda, strideA, a_dtype, a_layout};
  Operand Bop{B, ldb, strideB, b_dtype, b_layout};
  mpg_status s = validate(m, n, k, batch, Aop, Bop, C, ldc, strideC, alpha, mode, o);
  if (s != MPG_OK) return s;
  if (m == 0 || n == 0 || batch == 0) return MPG_OK;
  DeviceInfo* dev = nullptr;
  s = get_device(&dev);
  if (s != MPG_OK) return s;
  // A forced split count whose partial sums cannot fit the scratch is
  // refused here with a message naming the scratch; an automatic count is
  // left to the planner, which drops to one split when the partials do not
  // fit (as it does for a small caller workspace).
  if (o.splitk > 0 && k > 0 && alpha != 0.0f && mode != MPG_FP32_FFMA) {
    const size_t need = splitk_bytes(choose_splits(m, n, k, batch, dev->sm_count, o), m, n, batch);
    if (need > MPG_NOALLOC_SCRATCH_BYTES)
      return fail(MPG_ERR_WORKSPACE,
                  "split-K partial sums need %zu bytes, more than the %u-byte static scratch of "
                  "mpg_gemm_noalloc; call mpg_gemm with a workspace instead",
                  need, (unsigned)MPG_NOALLOC_SCRATCH_BYTES);
  }
  // The whole scratch is offered on every call, so that the planner sees
  // the same budget whatever the split count: the same plan as mpg_gemm_ex
  // given a workspace of MPG_NOALLOC_SCRATCH_BYTES.
  void* scratch = nullptr;
  s = noalloc_scratch(&scratch);
  if (s != MPG_OK) return s;
  // the split tail's partial sums would need more than the scratch holds
  // for the largest products: this entry never takes it
  o.tail_split = -1;
  return mpg_gemm_ex(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype, b_layout, C,
                     ldc, strideC, alpha, beta, mode, scratch, (size_t)MPG_NOALLOC_SCRATCH_BYTES, stream, &o);
}

}  // extern "C"
