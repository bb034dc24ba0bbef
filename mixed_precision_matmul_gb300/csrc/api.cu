// Host side of the C ABI: argument validation, plan selection (which kernel,
// tile width, split-K), TMA tensor-map encoding and launch.  Nothing here
// allocates device memory.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "internal.h"
#include "mpgemm.h"

namespace mpg {
bool tc_lookup_direct(Conv conv, Op op, int bn, TcKernel* out);
bool tc_lookup_staged(Conv conv, int bn, TcKernel* out);
bool tc_lookup_generic(Conv conv, Op op, SrcT st, int bn, TcKernel* out);

bool tc_kernel_lookup(Src src, Conv conv, Op op, SrcT st, int bn, TcKernel* out) {
  switch (src) {
    case Src::kTmaDirect: return tc_lookup_direct(conv, op, bn, out);
    case Src::kTmaStaged: return tc_lookup_staged(conv, bn, out);
    default: return tc_lookup_generic(conv, op, st, bn, out);
  }
}
}  // namespace mpg

using namespace mpg;

namespace {

thread_local std::string t_err;

mpg_status fail(mpg_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_err = buf;
  return s;
}

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
constexpr int64_t kDefaultSplitChunkK = 256;

struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int max_smem_optin = 0;
  uint32_t* status = nullptr;
  std::atomic<uint64_t> smem_set_mask[4];  // kernels whose smem attribute was set (by slot)
};

DeviceInfo g_devices[kMaxDevices];
std::mutex g_mu;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

mpg_status get_device(DeviceInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return fail(MPG_ERR_NO_DEVICE, "no CUDA device: %s", cudaGetErrorString(e));
  }
  if (dev >= kMaxDevices) return fail(MPG_ERR_NO_DEVICE, "device index %d beyond %d", dev, kMaxDevices);
  DeviceInfo& d = g_devices[dev];
  if (d.ready) {
    *out = &d;
    return MPG_OK;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) {
      return fail(MPG_ERR_NO_DEVICE, "device %d is sm_%d%d; this library is built for sm_103a only", dev, major,
                  minor);
    }
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    d.status = status_word_ptr();
    if (!d.status) return fail(MPG_ERR_CUDA, "cannot resolve the device status word");
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn) {
        cudaGetLastError();
        return fail(MPG_ERR_CUDA, "driver entry point cuTensorMapEncodeTiled unavailable");
      }
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    for (auto& m : d.smem_set_mask) m.store(0);
    d.ready = true;
  }
  *out = &d;
  return MPG_OK;
}

int elem_bytes(mpg_dtype t) { return t == MPG_F32 ? 4 : 2; }

// --------------------------------------------------------------------------
// planning
// --------------------------------------------------------------------------
enum class Kind { kNoop, kScale, kFfma, kTc };

struct Plan {
  Kind kind = Kind::kNoop;
  Src src = Src::kTmaDirect;
  Conv conv = Conv::kNone;
  Op op = Op::kF16;
  SrcT st = SrcT::kF32;
  int bn = 128;
  int splits = 1;
  bool prepass = false;       // operands converted by a separate pass into the workspace
  Conv pre_conv = Conv::kNone;
  bool pair = false;          // 256 x 256 tiles on CTA pairs (cta_group::2)
  bool copy_a = false;        // operand copied to an aligned layout in the workspace (TMA cannot
  bool copy_b = false;        //   describe it as given), then multiplied on the direct path
};

struct Operand {
  const void* ptr;
  int64_t ld, stride;
  mpg_dtype dt;
  mpg_layout layout;
};

bool tma_ok(const Operand& x, int64_t batch) {
  const int64_t es = elem_bytes(x.dt);
  if (reinterpret_cast<uintptr_t>(x.ptr) % 16 != 0) return false;
  if ((x.ld * es) % 16 != 0 || x.ld * es >= (int64_t(1) << 40)) return false;
  if (batch > 1 && ((x.stride * es) % 16 != 0 || x.stride * es >= (int64_t(1) << 40))) return false;
  return true;
}

// Number of K partitions from the sizes alone, so that the workspace query
// and the call agree whatever path the pointers select.  Counted with
// 128 x 128 tiles and 32-wide k-blocks.
int choose_splits(int64_t m, int64_t n, int64_t k, int64_t batch, int sm_count, const mpg_options& o) {
  const int64_t kb = (k + 31) / 32;
  if (o.splitk > 0) return (int)std::min<int64_t>(o.splitk, std::max<int64_t>(kb, 1));
  const int64_t tiles = batch * ((m + 127) / 128) * ((n + 127) / 128);
  if (tiles * 2 > sm_count || kb < 16) return 1;
  int64_t s = sm_count / tiles;
  s = std::min<int64_t>(s, kb / 8);
  return (int)std::max<int64_t>(s, 1);
}

size_t splitk_bytes(int splits, int64_t m, int64_t n, int64_t batch) {
  return splits > 1 ? (size_t)splits * (size_t)batch * (size_t)m * (size_t)n * sizeof(float) : 0;
}

// Workspace of the separate conversion pass: packed 16-bit copies of A and B
// (hi and lo for the split) after the split-K partials, each 256-byte aligned.
// A copy keeps its operand's majorness; its lines are padded to a multiple of
// 8 elements so that every line starts on a 16-byte boundary (TMA).
struct PrepassLayout {
  int64_t a_outer, a_inner, a_ld, b_outer, b_inner, b_ld;
  size_t off_a_hi, off_a_lo, off_b_hi, off_b_lo, end;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PrepassLayout prepass_layout(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_layout al, mpg_layout bl,
                             bool split_a, bool split_b, size_t base) {
  PrepassLayout L;
  L.a_outer = (al == MPG_ROW_MAJOR) ? m : k;
  L.a_inner = (al == MPG_ROW_MAJOR) ? k : m;
  L.b_outer = (bl == MPG_ROW_MAJOR) ? k : n;
  L.b_inner = (bl == MPG_ROW_MAJOR) ? n : k;
  L.a_ld = (L.a_inner + 7) / 8 * 8;
  L.b_ld = (L.b_inner + 7) / 8 * 8;
  const size_t a_bytes = align256((size_t)batch * L.a_outer * L.a_ld * 2);
  const size_t b_bytes = align256((size_t)batch * L.b_outer * L.b_ld * 2);
  size_t off = align256(base);
  L.off_a_hi = off; off += a_bytes;
  L.off_a_lo = off; off += split_a ? a_bytes : 0;
  L.off_b_hi = off; off += b_bytes;
  L.off_b_lo = off; off += split_b ? b_bytes : 0;
  L.end = off;
  return L;
}

// The split modes (fp32 inputs) take the separate conversion pass by
// default when both operands are re-read by many tiles: at least two
// 128-row tiles each way and 2^32 multiply-adds, where converting every
// operand element once in HBM costs far less than converting it in shared
// memory for every tile that reads it.
bool split_mode(mpg_precision mode) {
  return mode == MPG_SPLIT_FP16_3CHAIN || mode == MPG_SPLIT_FP16_1CHAIN || mode == MPG_SPLIT_A_FP16_2CHAIN ||
         mode == MPG_SPLIT_FP16_4CHAIN;
}
bool auto_prepass_shape(int64_t m, int64_t n, int64_t k) {
  return m >= 256 && n >= 256 && (double)m * (double)n * (double)k >= 4294967296.0;
}

// Workspace of the copies of operands the TMA path cannot take as given:
// dense copies in the operand's own type, in the layout the direct path
// needs (the source's own, or for tf32 A row-major and B column-major, whose
// tiles are K-major), lines padded to a multiple of 8 elements, after the
// split-K partials, 256-byte aligned.
struct CopyLayout {
  mpg_layout a_layout, b_layout;                 // layouts of the copies
  int64_t a_outer, a_inner, a_ld, b_outer, b_inner, b_ld;
  size_t off_a, off_b, end;
};

CopyLayout copy_layout(int64_t m, int64_t n, int64_t k, int64_t batch, const Operand& A, const Operand& B,
                       bool ca, bool cb, size_t base, mpg_layout a_out, mpg_layout b_out) {
  CopyLayout L;
  L.a_layout = a_out;
  L.b_layout = b_out;
  L.a_outer = (a_out == MPG_ROW_MAJOR) ? m : k;
  L.a_inner = (a_out == MPG_ROW_MAJOR) ? k : m;
  L.b_outer = (b_out == MPG_ROW_MAJOR) ? k : n;
  L.b_inner = (b_out == MPG_ROW_MAJOR) ? n : k;
  L.a_ld = (L.a_inner + 7) / 8 * 8;
  L.b_ld = (L.b_inner + 7) / 8 * 8;
  size_t off = align256(base);
  L.off_a = off;
  if (ca) off += align256((size_t)batch * L.a_outer * L.a_ld * elem_bytes(A.dt));
  L.off_b = off;
  if (cb) off += align256((size_t)batch * L.b_outer * L.b_ld * elem_bytes(B.dt));
  L.end = off;
  return L;
}

bool prepass_mode(mpg_precision mode) {
  return mode == MPG_FP16_F32ACC || mode == MPG_BF16_F32ACC || mode == MPG_SPLIT_FP16_3CHAIN ||
         mode == MPG_SPLIT_FP16_1CHAIN || mode == MPG_SPLIT_A_FP16_2CHAIN || mode == MPG_SPLIT_FP16_4CHAIN;
}

// Which operands carry hi and lo copies under a conversion.
bool splits_a(Conv c) {
  return c == Conv::kSplit3 || c == Conv::kSplit1 || c == Conv::kSplitA2 || c == Conv::kSplit4;
}
bool splits_b(Conv c) { return c == Conv::kSplit3 || c == Conv::kSplit1 || c == Conv::kSplit4; }

mpg_status make_plan(int64_t m, int64_t n, int64_t k, int64_t batch, const Operand& A, const Operand& B,
                     float alpha, mpg_precision mode, const mpg_options& o, int sm_count, size_t ws_bytes,
                     Plan* plan) {
  Plan p;
  if (m == 0 || n == 0 || batch == 0) {
    p.kind = Kind::kNoop;
    *plan = p;
    return MPG_OK;
  }
  if (k == 0 || alpha == 0.0f) {
    p.kind = Kind::kScale;
    *plan = p;
    return MPG_OK;
  }
  if (mode == MPG_FP32_FFMA) {
    p.kind = Kind::kFfma;
    *plan = p;
    return MPG_OK;
  }
  p.kind = Kind::kTc;
  const bool f32 = (A.dt == MPG_F32);
  bool direct_layout_ok = true;
  switch (mode) {
    case MPG_FP16_F32ACC:
      p.op = Op::kF16;
      p.conv = f32 ? Conv::kRoundF16 : Conv::kNone;
      p.st = f32 ? SrcT::kF32 : SrcT::kF16;
      break;
    case MPG_BF16_F32ACC:
      p.op = Op::kBF16;
      p.conv = f32 ? Conv::kRoundBF16 : Conv::kNone;
      p.st = f32 ? SrcT::kF32 : SrcT::kBF16;
      break;
    case MPG_TF32:
      p.op = Op::kTF32;
      p.conv = Conv::kNone;
      p.st = SrcT::kF32;
      // tf32 shared-memory tiles are kept K-major: the direct TMA path needs
      // a row-major A and a column-major B
      direct_layout_ok = (A.layout == MPG_ROW_MAJOR && B.layout == MPG_COL_MAJOR);
      break;
    case MPG_SPLIT_FP16_3CHAIN:
      p.op = Op::kF16;
      p.conv = Conv::kSplit3;
      p.st = SrcT::kF32;
      break;
    case MPG_SPLIT_FP16_1CHAIN:
      p.op = Op::kF16;
      p.conv = Conv::kSplit1;
      p.st = SrcT::kF32;
      break;
    case MPG_SPLIT_A_FP16_2CHAIN:
      p.op = Op::kF16;
      p.conv = Conv::kSplitA2;
      p.st = SrcT::kF32;
      break;
    case MPG_SPLIT_FP16_4CHAIN:
      p.op = Op::kF16;
      p.conv = Conv::kSplit4;
      p.st = SrcT::kF32;
      break;
    default:
      return fail(MPG_ERR_UNSUPPORTED, "unknown precision mode %d", (int)mode);
  }
  const bool tma = !o.force_generic_load && tma_ok(A, batch) && tma_ok(B, batch);
  // split-K is chosen from the sizes alone, before the path
  int splits = choose_splits(m, n, k, batch, sm_count, o);
  bool use_pass = (o.prepass == 1 && p.conv != Conv::kNone);
  // the library's choice: every mode that converts fp32 operands (split,
  // and fp16 / bf16 on fp32 inputs), when the workspace holds the copies
  // (the sizes-only query includes them for the split modes, the exact one
  // for all)
  if (!use_pass && o.prepass == 0 && p.conv != Conv::kNone && auto_prepass_shape(m, n, k)) {
    // the library's choice: the pass when the workspace holds the copies
    const PrepassLayout L = prepass_layout(m, n, k, batch, A.layout, B.layout, splits_a(p.conv), splits_b(p.conv),
                                           splitk_bytes(splits, m, n, batch));
    use_pass = (L.end <= ws_bytes);
  }
  if (use_pass) {
    // convert in a separate pass; the product reads packed 16-bit copies
    // (always TMA-aligned) on its direct path
    p.prepass = true;
    p.pre_conv = p.conv;
    p.src = Src::kTmaDirect;
    if (p.conv == Conv::kRoundF16 || p.conv == Conv::kRoundBF16) {
      p.conv = Conv::kNone;
      p.st = (p.op == Op::kBF16) ? SrcT::kBF16 : SrcT::kF16;
    } else {
      p.st = SrcT::kF16;
    }
  } else if (tma && p.conv == Conv::kNone && direct_layout_ok) {
    p.src = Src::kTmaDirect;
  } else if (tma && p.conv != Conv::kNone) {
    p.src = Src::kTmaStaged;
  } else {
    p.src = Src::kGeneric;
    // operands TMA cannot describe (unaligned base, leading dimension or
    // batch stride), and tf32 operands in the wrong majorness, are copied
    // to aligned lines in the layout the direct path needs when the
    // workspace holds the copies, then the direct path multiplies them
    if (!o.force_generic_load && p.conv == Conv::kNone) {
      const bool tf32 = (p.op == Op::kTF32);
      const mpg_layout a_out = tf32 ? MPG_ROW_MAJOR : A.layout;
      const mpg_layout b_out = tf32 ? MPG_COL_MAJOR : B.layout;
      const bool ca = !tma_ok(A, batch) || A.layout != a_out;
      const bool cb = !tma_ok(B, batch) || B.layout != b_out;
      const CopyLayout L =
          copy_layout(m, n, k, batch, A, B, ca, cb, splitk_bytes(splits, m, n, batch), a_out, b_out);
      if (L.end <= ws_bytes) {
        p.src = Src::kTmaDirect;
        p.copy_a = ca;
        p.copy_b = cb;
      }
    }
  }

  // tile width along N
  int bn;
  if (p.conv == Conv::kSplit4) {
    bn = 64;   // four chains of 64 columns plus the running sum fill TMEM
  } else if (p.src == Src::kGeneric) {
    bn = 128;
  } else if (p.src == Src::kTmaDirect && p.conv == Conv::kNone) {
    bn = n <= 64 ? 64 : (n <= 128 ? 128 : 256);
  } else if (p.conv == Conv::kSplit3 || p.conv == Conv::kSplitA2) {
    bn = (n <= 64 || k <= 512) ? 64 : 128;
  } else if (p.conv == Conv::kSplit1) {
    bn = n <= 64 ? 64 : 128;
  } else {
    // fp32 -> fp16 / bf16 on load: the widest tile converts the fewest
    // source bytes per flop
    bn = n <= 64 ? 64 : (n <= 128 ? 128 : 256);
  }
  if (o.tile_n != 0) {
    TcKernel probe;
    if (!tc_kernel_lookup(p.src, p.conv, p.op, p.st, o.tile_n, &probe))
      return fail(MPG_ERR_UNSUPPORTED, "tile_n %d is not available on this path", o.tile_n);
    bn = o.tile_n;
  }
  p.bn = bn;
  // CTA pairs: 16-bit operands on the direct path (also the conversion
  // pass's copies), 256 x 256 tiles.  Chosen by the library when those tiles
  // give every pair of SMs at least one (a smaller problem keeps the finer
  // 128-row tiles), or forced with cta_pair = 1.
  const bool pair_ok = p.src == Src::kTmaDirect && p.conv == Conv::kNone && p.op != Op::kTF32 &&
                       (o.tile_n == 0 || o.tile_n == 256);
  const int64_t pair_tiles = batch * ((m + 255) / 256) * ((n + 255) / 256);
  if (pair_ok && (o.cta_pair == 1 || (o.cta_pair == 0 && o.tile_n == 0 && pair_tiles * 2 >= sm_count))) {
    p.pair = true;
    p.bn = 256;
  }

  if (p.prepass) {
    const PrepassLayout L = prepass_layout(m, n, k, batch, A.layout, B.layout, splits_a(p.conv), splits_b(p.conv),
                                           splitk_bytes(splits, m, n, batch));
    if (L.end > ws_bytes)
      return fail(MPG_ERR_WORKSPACE, "the separate conversion pass needs %zu workspace bytes, got %zu", L.end,
                  ws_bytes);
  }
  if (splits > 1 && splitk_bytes(splits, m, n, batch) > ws_bytes) {
    if (o.splitk > 0)
      return fail(MPG_ERR_WORKSPACE, "split-K with %d partitions needs %zu workspace bytes, got %zu", splits,
                  splitk_bytes(splits, m, n, batch), ws_bytes);
    splits = 1;  // automatic choice: no workspace, no split
  }
  p.splits = splits;
  *plan = p;
  return MPG_OK;
}

// --------------------------------------------------------------------------
// validation
// --------------------------------------------------------------------------
mpg_status validate(int64_t m, int64_t n, int64_t k, int64_t batch, const Operand& A, const Operand& B,
                    const float* C, int64_t ldc, int64_t strideC, float alpha, mpg_precision mode,
                    const mpg_options& o) {
  const int64_t kMax = 0x7FFFFFFF;
  if (m < 0 || n < 0 || k < 0 || batch < 0)
    return fail(MPG_ERR_INVALID_ARG, "negative size (m=%lld n=%lld k=%lld batch=%lld)", (long long)m,
                (long long)n, (long long)k, (long long)batch);
  if (m > kMax || n > kMax || k > kMax || batch > kMax)
    return fail(MPG_ERR_INVALID_ARG, "size beyond 2^31-1");
  if ((int)mode < 0 || (int)mode > (int)MPG_SPLIT_FP16_4CHAIN)
    return fail(MPG_ERR_UNSUPPORTED, "unknown precision mode %d", (int)mode);
  for (const Operand* x : {&A, &B}) {
    if ((int)x->dt < 0 || (int)x->dt > 2) return fail(MPG_ERR_INVALID_ARG, "unknown dtype %d", (int)x->dt);
    if ((int)x->layout < 0 || (int)x->layout > 1) return fail(MPG_ERR_INVALID_ARG, "unknown layout %d", (int)x->layout);
  }
  if (A.dt != B.dt) return fail(MPG_ERR_UNSUPPORTED, "A and B must have the same dtype");
  switch (mode) {
    case MPG_FP16_F32ACC:
      if (A.dt != MPG_F32 && A.dt != MPG_F16) return fail(MPG_ERR_UNSUPPORTED, "FP16_F32ACC takes F32 or F16 inputs");
      break;
    case MPG_BF16_F32ACC:
      if (A.dt != MPG_F32 && A.dt != MPG_BF16) return fail(MPG_ERR_UNSUPPORTED, "BF16_F32ACC takes F32 or BF16 inputs");
      break;
    default:
      if (A.dt != MPG_F32) return fail(MPG_ERR_UNSUPPORTED, "this precision mode takes F32 inputs");
  }
  // leading dimensions (layout contract)
  const int64_t a_min = (A.layout == MPG_ROW_MAJOR) ? std::max<int64_t>(k, 1) : std::max<int64_t>(m, 1);
  const int64_t b_min = (B.layout == MPG_ROW_MAJOR) ? std::max<int64_t>(n, 1) : std::max<int64_t>(k, 1);
  if (A.ld < a_min) return fail(MPG_ERR_INVALID_ARG, "lda=%lld smaller than %lld", (long long)A.ld, (long long)a_min);
  if (B.ld < b_min) return fail(MPG_ERR_INVALID_ARG, "ldb=%lld smaller than %lld", (long long)B.ld, (long long)b_min);
  if (ldc < std::max<int64_t>(n, 1)) return fail(MPG_ERR_INVALID_ARG, "ldc=%lld smaller than n", (long long)ldc);
  if (A.stride < 0 || B.stride < 0 || strideC < 0) return fail(MPG_ERR_INVALID_ARG, "negative batch stride");
  if (o.split_exp_a < -100 || o.split_exp_a > 100 || o.split_exp_b < -100 || o.split_exp_b > 100)
    return fail(MPG_ERR_INVALID_ARG, "split exponent outside [-100, 100]");
  if (o.splitk < 0) return fail(MPG_ERR_INVALID_ARG, "negative splitk");
  if (o.wait_timeout_ns < 0) return fail(MPG_ERR_INVALID_ARG, "negative wait timeout");
  if (o.c_dtype < MPG_F32 || o.c_dtype > MPG_BF16) return fail(MPG_ERR_INVALID_ARG, "unknown C dtype %d", o.c_dtype);
  if (o.cta_pair < -1 || o.cta_pair > 1) return fail(MPG_ERR_INVALID_ARG, "cta_pair must be -1, 0 or 1");
  if (o.prepass < -1 || o.prepass > 1) return fail(MPG_ERR_INVALID_ARG, "prepass must be -1, 0 or 1");
  if (m == 0 || n == 0 || batch == 0) return MPG_OK;
  if (!C) return fail(MPG_ERR_INVALID_ARG, "C is NULL");
  if (reinterpret_cast<uintptr_t>(C) % (o.c_dtype == MPG_F32 ? 4 : 2) != 0)
    return fail(MPG_ERR_INVALID_ARG, "C not aligned to its element size");
  if (k > 0 && alpha != 0.0f) {
    if (!A.ptr || !B.ptr) return fail(MPG_ERR_INVALID_ARG, "A or B is NULL");
    if (reinterpret_cast<uintptr_t>(A.ptr) % elem_bytes(A.dt) != 0 ||
        reinterpret_cast<uintptr_t>(B.ptr) % elem_bytes(B.dt) != 0)
      return fail(MPG_ERR_INVALID_ARG, "A or B not aligned to its element size");
  }
  return MPG_OK;
}

void resolve_options(const mpg_options* opt, mpg_options* o) {
  mpg_options_init(o);
  if (opt) *o = *opt;
}

CUtensorMapDataType tma_dtype(mpg_dtype t) {
  return t == MPG_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                      : (t == MPG_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// 3-D map {inner, outer, batch}, box {box_inner, box_outer, 1}, 128B swizzle.
mpg_status encode_map(CUtensorMap* map, const Operand& x, int64_t inner, int64_t outer, int64_t batch,
                      int box_inner, int box_outer) {
  const int64_t es = elem_bytes(x.dt);
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)std::max<int64_t>(batch, 1)};
  cuuint64_t strides[2] = {(cuuint64_t)(x.ld * es),
                           (cuuint64_t)(batch > 1 ? x.stride * es : x.ld * es * std::max<int64_t>(outer, 1))};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, tma_dtype(x.dt), 3, const_cast<void*>(x.ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MPG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MPG_OK;
}

// Clusters of two CTAs of the pair kernel that fit on the device at once,
// asked once per device (both pair kernels have the same launch shape).
mpg_status pair_clusters(DeviceInfo* dev, const TcKernel& kern, int* out) {
  static std::mutex mu;
  static int cached[kMaxDevices];
  const int devid = (int)(dev - g_devices);
  std::lock_guard<std::mutex> lock(mu);
  if (cached[devid] <= 0) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3((unsigned)kern.block);
    cfg.dynamicSmemBytes = (size_t)kern.smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kern.fn, &cfg);
    if (e != cudaSuccess || n < 1) {
      cudaGetLastError();
      return fail(MPG_ERR_UNSUPPORTED, "no resident cluster of two CTAs for the pair kernel: %s",
                  e != cudaSuccess ? cudaGetErrorString(e) : "occupancy 0");
    }
    cached[devid] = n;
  }
  *out = cached[devid];
  return MPG_OK;
}

mpg_status launch_tc(const Plan& plan, DeviceInfo* dev, int64_t m, int64_t n, int64_t k, int64_t batch,
                     const Operand& A, const Operand& B, float* C, int64_t ldc, int64_t strideC, float alpha,
                     float beta, const mpg_options& o, void* workspace, cudaStream_t stream,
                     const Operand* A_lo = nullptr, const Operand* B_lo = nullptr) {
  TcKernel kern;
  const bool found = plan.pair ? mpg::tc_lookup_pair(plan.op, &kern)
                               : mpg::tc_kernel_lookup(plan.src, plan.conv, plan.op, plan.st, plan.bn, &kern);
  if (!found) return fail(MPG_ERR_UNSUPPORTED, "no kernel for this configuration");
  if (kern.smem_bytes > dev->max_smem_optin)
    return fail(MPG_ERR_UNSUPPORTED, "kernel needs %d bytes of shared memory, device offers %d", kern.smem_bytes,
                dev->max_smem_optin);
  // the dynamic shared-memory attribute is set once per kernel per device
  {
    const uintptr_t key = reinterpret_cast<uintptr_t>(kern.fn);
    static std::mutex attr_mu;
    static const void* done[kMaxDevices][64];
    static int ndone[kMaxDevices];
    int devid = (int)(dev - g_devices);
    std::lock_guard<std::mutex> lock(attr_mu);
    bool found = false;
    for (int i = 0; i < ndone[devid]; ++i)
      if (reinterpret_cast<uintptr_t>(done[devid][i]) == key) found = true;
    if (!found) {
      cudaError_t e = cudaFuncSetAttribute(kern.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kern.smem_bytes);
      if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "cudaFuncSetAttribute: %s", cudaGetErrorString(e));
      if (ndone[devid] < 64) done[devid][ndone[devid]++] = kern.fn;
    }
  }

  TcParams p;
  std::memset(&p, 0, sizeof(p));
  const int BK = (plan.src == Src::kTmaDirect) ? (plan.op == Op::kTF32 ? 32 : 64) : 32;
  const int BM = plan.pair ? 256 : 128;   // rows of C per tile (a pair: 128 per CTA)
  const int bn = plan.bn;
  const int a_box = 128;                  // rows of A per CTA
  const int b_box = plan.pair ? bn / 2 : bn;   // rows of a K-major B tile per CTA
  const bool a_mn = (A.layout == MPG_COL_MAJOR);
  const bool b_mn = (B.layout == MPG_ROW_MAJOR);
  const int64_t a_stride = A.stride ? A.stride : (a_mn ? k * A.ld : m * A.ld);
  const int64_t b_stride = B.stride ? B.stride : (b_mn ? k * B.ld : n * B.ld);
  Operand Ax = A, Bx = B;
  Ax.stride = a_stride;
  Bx.stride = b_stride;
  if (plan.src != Src::kGeneric) {
    mpg_status s;
    // staged path: fp32 boxes of 32 elements (128 bytes) per line
    if (!a_mn) s = encode_map(&p.map_a, Ax, k, m, batch, BK, a_box);
    else s = encode_map(&p.map_a, Ax, m, k, batch, BK, BK);
    if (s != MPG_OK) return s;
    if (!b_mn) s = encode_map(&p.map_b, Bx, k, n, batch, BK, b_box);
    else s = encode_map(&p.map_b, Bx, n, k, batch, BK, BK);
    if (s != MPG_OK) return s;
    // lo halves of pre-split operands: same geometry as the hi halves
    if (A_lo) {
      Operand Al = *A_lo;
      Al.stride = a_stride;
      if (!a_mn) s = encode_map(&p.map_a_lo, Al, k, m, batch, BK, a_box);
      else s = encode_map(&p.map_a_lo, Al, m, k, batch, BK, BK);
      if (s != MPG_OK) return s;
    }
    if (B_lo) {
      Operand Bl = *B_lo;
      Bl.stride = b_stride;
      if (!b_mn) s = encode_map(&p.map_b_lo, Bl, k, n, batch, BK, b_box);
      else s = encode_map(&p.map_b_lo, Bl, n, k, batch, BK, BK);
      if (s != MPG_OK) return s;
    }
  }
  p.a = A.ptr;
  p.b = B.ptr;
  p.lda = A.ld;
  p.ldb = B.ld;
  p.stride_a = a_stride;
  p.stride_b = b_stride;
  p.c = C;
  p.ldc = ldc;
  p.stride_c = strideC ? strideC : m * ldc;
  p.m = (int32_t)m;
  p.n = (int32_t)n;
  p.k = (int32_t)k;
  p.batch = (int32_t)batch;
  p.a_mn_major = a_mn;
  p.b_mn_major = b_mn;
  p.num_m_blk = (int32_t)((m + BM - 1) / BM);
  p.num_n_blk = (int32_t)((n + bn - 1) / bn);
  p.num_k_blk = (int32_t)((k + BK - 1) / BK);
  int kb_per = (p.num_k_blk + plan.splits - 1) / plan.splits;
  int splits_eff = (p.num_k_blk + kb_per - 1) / kb_per;
  p.splits = splits_eff;
  p.kb_per_split = kb_per;
  const int64_t tiles = (int64_t)splits_eff * batch * p.num_m_blk * p.num_n_blk;
  if (tiles > 0x7FFFFFFF) return fail(MPG_ERR_INVALID_ARG, "too many tiles");
  p.num_tiles = (int32_t)tiles;
  // rasterisation: groups of tile rows sized so that the tiles resident at
  // once touch about as many A panels as B panels (tiles of a pair are
  // twice as tall)
  p.group_m = plan.pair ? 8 : 16;
  p.c_dtype = o.c_dtype;
  p.c_vec_ok = (reinterpret_cast<uintptr_t>(C) % (o.c_dtype == MPG_F32 ? 16 : 8) == 0) && (ldc % 4 == 0) &&
               (batch == 1 || p.stride_c % 4 == 0);
  // generic loads read 4 consecutive elements as one vector when the base,
  // the leading dimension and the batch stride keep every chunk aligned
  auto vec_ok = [&](const Operand& x, int64_t stride) {
    const int64_t es = elem_bytes(x.dt);
    return reinterpret_cast<uintptr_t>(x.ptr) % (4 * es) == 0 && x.ld % 4 == 0 &&
           (batch == 1 || stride % 4 == 0);
  };
  p.a_vec_ok = vec_ok(A, a_stride);
  p.b_vec_ok = vec_ok(B, b_stride);
  p.partial = splits_eff > 1 ? static_cast<float*>(workspace) : nullptr;
  p.p_vec_ok = (n % 4 == 0) && (reinterpret_cast<uintptr_t>(workspace) % 16 == 0);
  const bool split = splits_a(plan.conv);
  const int sa = split ? o.split_exp_a : 0, sb = split ? o.split_exp_b : 0;
  p.alpha = (float)std::ldexp((double)alpha, -(sa + sb));
  p.beta = beta;
  p.scale_a = std::ldexp(1.0f, sa);
  p.scale_b = std::ldexp(1.0f, sb);
  p.status = dev->status;
  p.wait_limit_ns = o.wait_timeout_ns > 0 ? (uint64_t)o.wait_timeout_ns : kDefaultWaitNs;
  p.chunk_kb = 0;
  if ((plan.conv == Conv::kSplit3 || plan.conv == Conv::kSplitA2 || plan.conv == Conv::kSplit4) &&
      o.split_chunk_k >= 0) {
    const int64_t chunk_k = o.split_chunk_k > 0 ? o.split_chunk_k : kDefaultSplitChunkK;
    p.chunk_kb = (int32_t)std::min<int64_t>((chunk_k + BK - 1) / BK, p.num_k_blk);
  }

  void* args[] = {&p};
  cudaError_t e;
  if (plan.pair) {
    // clusters of two CTAs; as many clusters as can be resident at once
    int clusters = 0;
    mpg_status cs = pair_clusters(dev, kern, &clusters);
    if (cs != MPG_OK) return cs;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)(2 * std::min<int64_t>(tiles, clusters)));
    cfg.blockDim = dim3((unsigned)kern.block);
    cfg.dynamicSmemBytes = (size_t)kern.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelExC(&cfg, kern.fn, args);
  } else {
    const int grid = (int)std::min<int64_t>(tiles, dev->sm_count);
    e = cudaLaunchKernel(kern.fn, dim3(grid), dim3(kern.block), args, kern.smem_bytes, stream);
  }
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  if (splits_eff > 1) {
    // the reduction applies alpha (incl. the split scale) and beta
    e = launch_splitk_reduce(p.partial, splits_eff, C, o.c_dtype, ldc, p.stride_c, p.m, p.n, p.batch, p.alpha, beta,
                             stream);
    if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "split-K reduce launch: %s", cudaGetErrorString(e));
  }
  return MPG_OK;
}

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

// --------------------------------------------------------------------------
// host-buffer entry point: device copies, chunk plan, internal streams
// --------------------------------------------------------------------------
// Stored footprint of one operand: `batch` matrices of `outer` lines of
// `inner` elements, lines `ld` apart, matrices `stride` apart.
struct Footprint {
  int64_t outer = 0, inner = 0, ld = 0, stride = 0, batch = 0, es = 0;
  // elements from the first to the last stored element (padding between
  // lines included, nothing past the last element)
  int64_t span() const { return (batch == 0 || outer == 0) ? 0 : (batch - 1) * stride + (outer - 1) * ld + inner; }
};

constexpr int kMaxHostChunks = 8;
constexpr int64_t kHostChunkBytes = int64_t(64) << 20;   // input bytes per chunk, about

// Host operands keep the caller's leading dimensions and batch strides; their
// device copies are packed with lines padded to 16 bytes (A and B to
// multiples of 8 elements, C to 4 fp32 or 8 16-bit elements), so the product
// always takes the TMA path whatever the host layout.
struct HostPlan {
  Footprint ha, hb, hc;    // host
  Footprint da, db, dc;    // device copies
  bool need_ab = false;    // A and B are read (k > 0, alpha != 0)
  bool need_c0 = false;    // C is read (beta != 0)
  bool by_batch = false;   // chunks of whole matrices (batch > 1), else of rows of A and C
  int64_t chunk = 0;       // rows, or matrices, per chunk
  int nchunks = 0;
  size_t off_a = 0, off_b = 0, off_c = 0, off_ws = 0, ws_bytes = 0, total = 0;
};

Footprint device_copy(const Footprint& h, int64_t align) {
  Footprint d = h;
  d.ld = std::max<int64_t>(align, (h.inner + align - 1) / align * align);   // >= 1 also for empty lines
  d.stride = h.outer * d.ld;
  return d;
}

mpg_status host_plan(int64_t m, int64_t n, int64_t k, int64_t batch, int64_t lda, int64_t strideA, mpg_dtype adt,
                     mpg_layout al, int64_t ldb, int64_t strideB, mpg_dtype bdt, mpg_layout bl, int64_t ldc,
                     int64_t strideC, float alpha, float beta, mpg_precision mode, const mpg_options& o,
                     HostPlan* out) {
  HostPlan h;
  const bool a_row = (al == MPG_ROW_MAJOR), b_row = (bl == MPG_ROW_MAJOR);
  const int64_t ces = (o.c_dtype == MPG_F32) ? 4 : 2;
  h.ha = {a_row ? m : k, a_row ? k : m, lda, 0, batch, elem_bytes(adt)};
  h.hb = {b_row ? k : n, b_row ? n : k, ldb, 0, batch, elem_bytes(bdt)};
  h.hc = {m, n, ldc, 0, batch, ces};
  h.ha.stride = strideA ? strideA : h.ha.outer * lda;
  h.hb.stride = strideB ? strideB : h.hb.outer * ldb;
  h.hc.stride = strideC ? strideC : m * ldc;
  h.da = device_copy(h.ha, 8);
  h.db = device_copy(h.hb, 8);
  h.dc = device_copy(h.hc, ces == 4 ? 4 : 8);
  h.need_ab = (k > 0 && alpha != 0.0f);
  h.need_c0 = (beta != 0.0f);
  const int64_t in_bytes = (h.need_ab ? h.da.span() * h.da.es : 0) + (h.need_c0 ? h.dc.span() * h.dc.es : 0);
  int64_t want = std::min<int64_t>(kMaxHostChunks, std::max<int64_t>(1, in_bytes / kHostChunkBytes));
  h.by_batch = batch > 1;
  if (h.by_batch) {
    want = std::min<int64_t>(want, batch);
    h.chunk = (batch + want - 1) / want;
    h.nchunks = (int)((batch + h.chunk - 1) / h.chunk);
  } else {
    // row chunks in multiples of 256 rows (a whole number of tiles)
    want = std::min<int64_t>(want, std::max<int64_t>(1, m / 256));
    h.chunk = ((m + want - 1) / want + 255) / 256 * 256;
    h.nchunks = (int)((m + h.chunk - 1) / h.chunk);
  }
  // product workspace on the device copies (aligned: the 256 below only
  // stands for an aligned address): the larger of a full chunk and the last
  auto ws_for = [&](int64_t units) {
    const void* aligned = reinterpret_cast<const void*>(uintptr_t(256));
    return h.by_batch
               ? mpg_gemm_workspace_size_ex(m, n, k, units, aligned, h.da.ld, h.da.stride, adt, al, aligned, h.db.ld,
                                            h.db.stride, bdt, bl, mode, &o)
               : mpg_gemm_workspace_size_ex(units, n, k, 1, aligned, h.da.ld, 0, adt, al, aligned, h.db.ld, 0, bdt,
                                            bl, mode, &o);
  };
  const int64_t total_units = h.by_batch ? batch : m;
  const int64_t last = total_units - (int64_t)(h.nchunks - 1) * h.chunk;
  h.ws_bytes = std::max(ws_for(h.chunk), ws_for(last));
  size_t off = 0;
  h.off_a = off; off += align256((size_t)(h.need_ab ? h.da.span() * h.da.es : 0));
  h.off_b = off; off += align256((size_t)(h.need_ab ? h.db.span() * h.db.es : 0));
  h.off_c = off; off += align256((size_t)(h.dc.span() * h.dc.es));
  h.off_ws = off; off += align256(h.ws_bytes);
  h.total = off;
  *out = h;
  return MPG_OK;
}

// Internal copy streams of one device and the events that order them against
// the caller's stream.  One call enqueues at a time (the mutex).
struct HostStreams {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t ev[2 + 2 * kMaxHostChunks] = {};
  std::mutex mu;
};
HostStreams g_host[kMaxDevices];

mpg_status host_streams(HostStreams** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return fail(MPG_ERR_NO_DEVICE, "no current CUDA device");
  }
  HostStreams& hs = g_host[dev];
  std::lock_guard<std::mutex> lock(g_mu);
  if (!hs.ready) {
    cudaError_t e = cudaStreamCreateWithFlags(&hs.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&hs.out, cudaStreamNonBlocking);
    for (auto& ev : hs.ev)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "copy streams: %s", cudaGetErrorString(e));
    hs.ready = true;
  }
  *out = &hs;
  return MPG_OK;
}

// Lines [l0, l1) of matrices [b0, b1) of one operand, `width` elements of
// each line starting at element c0, from `src` laid out as fs to `dst` laid
// out as fd (the same matrices, different leading dimensions and strides).
cudaError_t copy_lines(const Footprint& fd, void* dst, const Footprint& fs, const void* src, int64_t b0, int64_t b1,
                       int64_t l0, int64_t l1, int64_t c0, int64_t width, cudaMemcpyKind kind, cudaStream_t st) {
  const int64_t lines = l1 - l0;
  if (lines <= 0 || b1 <= b0 || width <= 0) return cudaSuccess;
  const int64_t es = fs.es;
  auto at = [&](const Footprint& f, const void* base, int64_t b) {
    return static_cast<const uint8_t*>(base) + ((b * f.stride + l0 * f.ld + c0) * es);
  };
  const bool whole = (l0 == 0 && l1 == fs.outer);
  if (b1 - b0 == 1 || (whole && fs.stride == fs.outer * fs.ld && fd.stride == fd.outer * fd.ld)) {
    // one run of equally spaced lines on both sides
    const int64_t rows = (b1 - b0 == 1) ? lines : (b1 - b0) * fs.outer;
    return cudaMemcpy2DAsync(const_cast<uint8_t*>(at(fd, dst, b0)), (size_t)(fd.ld * es), at(fs, src, b0),
                             (size_t)(fs.ld * es), (size_t)(width * es), (size_t)rows, kind, st);
  }
  for (int64_t b = b0; b < b1; ++b) {
    cudaError_t e = cudaMemcpy2DAsync(const_cast<uint8_t*>(at(fd, dst, b)), (size_t)(fd.ld * es), at(fs, src, b),
                                      (size_t)(fs.ld * es), (size_t)(width * es), (size_t)lines, kind, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// --------------------------------------------------------------------------
// fused attention: key ranges and workspace
// --------------------------------------------------------------------------
struct AttnSplit {
  int splits = 1, kb_per_split = 1;
  size_t off_m = 0, off_l = 0, bytes = 0;
};

AttnSplit attention_split(int64_t lq, int64_t lk, int32_t key_splits, int sm_count) {
  AttnSplit a;
  const int64_t nkb = (lk + 63) / 64;
  const int64_t nqb = (lq + 127) / 128;
  int64_t s = key_splits > 0 ? key_splits : std::max<int64_t>(1, sm_count / std::max<int64_t>(nqb, 1));
  s = std::max<int64_t>(1, std::min<int64_t>(s, nkb));
  a.kb_per_split = (int)((nkb + s - 1) / s);
  a.splits = (int)((nkb + a.kb_per_split - 1) / a.kb_per_split);
  if (a.splits > 1) {
    const size_t o_bytes = align256((size_t)a.splits * (size_t)lq * 128 * sizeof(float));
    const size_t v_bytes = align256((size_t)a.splits * (size_t)lq * sizeof(float));
    a.off_m = o_bytes;
    a.off_l = o_bytes + v_bytes;
    a.bytes = o_bytes + 2 * v_bytes;
  }
  return a;
}

}  // namespace

extern "C" {

void mpg_options_init(mpg_options* opt) {
  if (!opt) return;
  std::memset(opt, 0, sizeof(*opt));
}

int mpg_version(void) { return 100; }

const char* mpg_last_error_string(void) { return t_err.c_str(); }

size_t mpg_gemm_workspace_size(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_precision mode,
                               const mpg_options* opt) {
  mpg_options o;
  resolve_options(opt, &o);
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0 || mode == MPG_FP32_FFMA) return 0;
  DeviceInfo* dev = nullptr;
  int sm = 152;
  if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
  t_err.clear();
  const size_t partials = splitk_bytes(choose_splits(m, n, k, batch, sm, o), m, n, batch);
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

size_t mpg_gemm_workspace_size_ex(int64_t m, int64_t n, int64_t k, int64_t batch, const void* A, int64_t lda,
                                  int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout, const void* B,
                                  int64_t ldb, int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout,
                                  mpg_precision mode, const mpg_options* opt) {
  mpg_options o;
  resolve_options(opt, &o);
  const size_t base = mpg_gemm_workspace_size(m, n, k, batch, mode, opt);
  if (m <= 0 || n <= 0 || k <= 0 || batch <= 0 || o.force_generic_load) return base;
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
    return std::max(base, L.end);
  }
  if (!f16in && !tf32) return base;
  Operand Aop{A, lda, strideA, a_dtype, a_layout};
  Operand Bop{B, ldb, strideB, b_dtype, b_layout};
  const mpg_layout a_out = tf32 ? MPG_ROW_MAJOR : a_layout, b_out = tf32 ? MPG_COL_MAJOR : b_layout;
  const bool ca = !tma_ok(Aop, batch) || a_layout != a_out, cb = !tma_ok(Bop, batch) || b_layout != b_out;
  if (!ca && !cb) return base;
  DeviceInfo* dev = nullptr;
  int sm = 152;
  if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
  t_err.clear();
  const CopyLayout L = copy_layout(m, n, k, batch, Aop, Bop, ca, cb,
                                   splitk_bytes(choose_splits(m, n, k, batch, sm, o), m, n, batch), a_out, b_out);
  return std::max(base, L.end);
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
        return launch_tc(plan, dev, m, n, k, batch, Ac, Bc, C, ldc, strideC, alpha, beta, o, workspace, st);
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
      const Conv conv_a = (plan.pre_conv == Conv::kSplitA2 || plan.pre_conv == Conv::kSplit4) ? Conv::kSplit3
                                                                                              : plan.pre_conv;
      const Conv conv_b = (plan.pre_conv == Conv::kSplitA2)  ? Conv::kRoundF16
                          : (plan.pre_conv == Conv::kSplit4) ? Conv::kSplit3
                                                             : plan.pre_conv;
      const int64_t sA = strideA ? strideA : L.a_outer * lda;
      const int64_t sB = strideB ? strideB : L.b_outer * ldb;
      e = launch_prepass(conv_a, static_cast<const float*>(A), lda, sA, L.a_outer, L.a_inner, batch, a_hi, a_lo,
                         L.a_ld, std::ldexp(1.0f, ea), dev->sm_count, st);
      if (e == cudaSuccess)
        e = launch_prepass(conv_b, static_cast<const float*>(B), ldb, sB, L.b_outer, L.b_inner, batch, b_hi, b_lo,
                           L.b_ld, std::ldexp(1.0f, eb), dev->sm_count, st);
      if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "conversion pass launch: %s", cudaGetErrorString(e));
      const mpg_dtype cdt = (plan.op == Op::kBF16) ? MPG_BF16 : MPG_F16;
      Operand Ah{a_hi, L.a_ld, L.a_outer * L.a_ld, cdt, a_layout};
      Operand Bh{b_hi, L.b_ld, L.b_outer * L.b_ld, cdt, b_layout};
      Operand Al{a_lo, L.a_ld, L.a_outer * L.a_ld, cdt, a_layout};
      Operand Bl{b_lo, L.b_ld, L.b_outer * L.b_ld, cdt, b_layout};
      return launch_tc(plan, dev, m, n, k, batch, Ah, Bh, C, ldc, strideC, alpha, beta, o, workspace, st,
                       sa_ ? &Al : nullptr, sb_ ? &Bl : nullptr);
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
  // the split-K scratch this problem needs (the same choice mpg_gemm makes)
  size_t need = 0;
  if (k > 0 && alpha != 0.0f && mode != MPG_FP32_FFMA)
    need = splitk_bytes(choose_splits(m, n, k, batch, dev->sm_count, o), m, n, batch);
  if (need > MPG_NOALLOC_SCRATCH_BYTES)
    return fail(MPG_ERR_WORKSPACE,
                "split-K partial sums need %zu bytes, more than the %u-byte static scratch of "
                "mpg_gemm_noalloc; call mpg_gemm with a workspace instead",
                need, (unsigned)MPG_NOALLOC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (need > 0) {
    s = noalloc_scratch(&scratch);
    if (s != MPG_OK) return s;
  }
  return mpg_gemm_ex(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype, b_layout, C,
                     ldc, strideC, alpha, beta, mode, scratch, need > 0 ? (size_t)MPG_NOALLOC_SCRATCH_BYTES : 0,
                     stream, opt);
}

size_t mpg_gemm_host_workspace_size(int64_t m, int64_t n, int64_t k, int64_t batch, int64_t lda, int64_t strideA,
                                    mpg_dtype a_dtype, mpg_layout a_layout, int64_t ldb, int64_t strideB,
                                    mpg_dtype b_dtype, mpg_layout b_layout, int64_t ldc, int64_t strideC,
                                    float alpha, float beta, mpg_precision mode, const mpg_options* opt) {
  mpg_options o;
  resolve_options(opt, &o);
  if (m <= 0 || n <= 0 || batch <= 0 || k < 0) return 0;
  HostPlan h;
  if (host_plan(m, n, k, batch, lda, strideA, a_dtype, a_layout, ldb, strideB, b_dtype, b_layout, ldc, strideC,
                alpha, beta, mode, o, &h) != MPG_OK)
    return 0;
  t_err.clear();
  return h.total;
}

mpg_status mpg_gemm_host(int64_t m, int64_t n, int64_t k, int64_t batch, const void* A, int64_t lda,
                         int64_t strideA, mpg_dtype a_dtype, mpg_layout a_layout, const void* B, int64_t ldb,
                         int64_t strideB, mpg_dtype b_dtype, mpg_layout b_layout, void* C, int64_t ldc,
                         int64_t strideC, float alpha, float beta, mpg_precision mode, void* workspace,
                         size_t workspace_bytes, void* stream, const mpg_options* opt) {
  t_err.clear();
  mpg_options o;
  resolve_options(opt, &o);
  Operand Aop{A, lda, strideA, a_dtype, a_layout};
  Operand Bop{B, ldb, strideB, b_dtype, b_layout};
  mpg_status s = validate(m, n, k, batch, Aop, Bop, static_cast<const float*>(C), ldc, strideC, alpha, mode, o);
  if (s != MPG_OK) return s;
  if (m == 0 || n == 0 || batch == 0) return MPG_OK;
  HostPlan h;
  s = host_plan(m, n, k, batch, lda, strideA, a_dtype, a_layout, ldb, strideB, b_dtype, b_layout, ldc, strideC,
                alpha, beta, mode, o, &h);
  if (s != MPG_OK) return s;
  if (!workspace || reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
    return fail(MPG_ERR_INVALID_ARG, "workspace missing or not 16-byte aligned");
  if (workspace_bytes < h.total)
    return fail(MPG_ERR_WORKSPACE, "host-buffer product needs %zu workspace bytes, got %zu", h.total,
                workspace_bytes);
  HostStreams* hs = nullptr;
  s = host_streams(&hs);
  if (s != MPG_OK) return s;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* dA = ws + h.off_a;
  uint8_t* dB = ws + h.off_b;
  uint8_t* dC = ws + h.off_c;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::lock_guard<std::mutex> lock(hs->mu);
  cudaEvent_t ev_start = hs->ev[0], ev_end = hs->ev[1];
  // copies start once earlier work of the caller's stream (which may still
  // use this workspace) is done
  cudaError_t e = cudaEventRecord(ev_start, st);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->in, ev_start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->out, ev_start, 0);
  if (e == cudaSuccess && h.need_ab)
    e = copy_lines(h.db, dB, h.hb, B, 0, batch, 0, h.hb.outer, 0, h.hb.inner, cudaMemcpyHostToDevice, hs->in);
  mpg_status prod = MPG_OK;
  const bool a_row = (a_layout == MPG_ROW_MAJOR);
  const int64_t es_a = h.da.es, es_b = h.db.es, es_c = h.dc.es;
  for (int c = 0; c < h.nchunks && e == cudaSuccess && prod == MPG_OK; ++c) {
    cudaEvent_t ev_in = hs->ev[2 + 2 * c], ev_cmp = hs->ev[3 + 2 * c];
    const int64_t u0 = (int64_t)c * h.chunk;
    const int64_t u1 = std::min<int64_t>(h.by_batch ? batch : m, u0 + h.chunk);
    // ---- inputs of the chunk
    if (h.by_batch) {
      if (h.need_ab)
        e = copy_lines(h.da, dA, h.ha, A, u0, u1, 0, h.ha.outer, 0, h.ha.inner, cudaMemcpyHostToDevice, hs->in);
      if (e == cudaSuccess && h.need_c0)
        e = copy_lines(h.dc, dC, h.hc, C, u0, u1, 0, m, 0, n, cudaMemcpyHostToDevice, hs->in);
    } else {
      if (h.need_ab) {
        if (a_row) e = copy_lines(h.da, dA, h.ha, A, 0, 1, u0, u1, 0, k, cudaMemcpyHostToDevice, hs->in);
        else e = copy_lines(h.da, dA, h.ha, A, 0, 1, 0, k, u0, u1 - u0, cudaMemcpyHostToDevice, hs->in);
      }
      if (e == cudaSuccess && h.need_c0)
        e = copy_lines(h.dc, dC, h.hc, C, 0, 1, u0, u1, 0, n, cudaMemcpyHostToDevice, hs->in);
    }
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, hs->in);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(st, ev_in, 0);
    if (e != cudaSuccess) break;
    // ---- the chunk's product on the caller's stream, on the device copies
    if (h.by_batch) {
      prod = mpg_gemm_ex(m, n, k, u1 - u0, dA + u0 * h.da.stride * es_a, h.da.ld, h.da.stride, a_dtype, a_layout,
                         dB + u0 * h.db.stride * es_b, h.db.ld, h.db.stride, b_dtype, b_layout,
                         reinterpret_cast<float*>(dC + u0 * h.dc.stride * es_c), h.dc.ld, h.dc.stride, alpha, beta,
                         mode, ws + h.off_ws, h.ws_bytes, st, &o);
    } else {
      const int64_t a_off = a_row ? u0 * h.da.ld : u0;
      prod = mpg_gemm_ex(u1 - u0, n, k, 1, dA + a_off * es_a, h.da.ld, 0, a_dtype, a_layout, dB, h.db.ld, 0, b_dtype,
                         b_layout, reinterpret_cast<float*>(dC + u0 * h.dc.ld * es_c), h.dc.ld, 0, alpha, beta, mode,
                         ws + h.off_ws, h.ws_bytes, st, &o);
    }
    if (prod != MPG_OK) break;
    e = cudaEventRecord(ev_cmp, st);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->out, ev_cmp, 0);
    // ---- the chunk's C back to the host (n elements of each row: C's
    //      padding columns are never written)
    if (e == cudaSuccess) {
      if (h.by_batch) e = copy_lines(h.hc, C, h.dc, dC, u0, u1, 0, m, 0, n, cudaMemcpyDeviceToHost, hs->out);
      else e = copy_lines(h.hc, C, h.dc, dC, 0, 1, u0, u1, 0, n, cudaMemcpyDeviceToHost, hs->out);
    }
  }
  // the caller's stream continues after the last copy back, also on error
  cudaError_t e2 = cudaEventRecord(ev_end, hs->out);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st, ev_end, 0);
  if (prod != MPG_OK) return prod;
  if (e == cudaSuccess) e = e2;
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "host-buffer product: %s", cudaGetErrorString(e));
  return MPG_OK;
}

size_t mpg_attention_workspace_size(int64_t lq, int64_t lk, int64_t d, int32_t key_splits) {
  if (lq <= 0 || lk <= 0 || d != 128 || key_splits < 0) return 0;
  DeviceInfo* dev = nullptr;
  int sm = 152;
  if (get_device(&dev) == MPG_OK) sm = dev->sm_count;
  t_err.clear();
  return attention_split(lq, lk, key_splits, sm).bytes;
}

mpg_status mpg_attention(int64_t lq, int64_t lk, int64_t d, const float* Q, int64_t ldq, const void* K, int64_t ldk,
                         const void* V, int64_t ldv, float* O, int64_t ldo, float scale, mpg_attn_mode mode,
                         int32_t key_splits, void* workspace, size_t workspace_bytes, void* stream) {
  t_err.clear();
  if (lq < 0 || lk < 0 || d < 0) return fail(MPG_ERR_INVALID_ARG, "negative size");
  if (lq > 0x7FFFFFFF || lk > 0x7FFFFFFF) return fail(MPG_ERR_INVALID_ARG, "size beyond 2^31-1");
  if ((int)mode < 0 || (int)mode > 1) return fail(MPG_ERR_UNSUPPORTED, "unknown attention mode %d", (int)mode);
  if (key_splits < 0) return fail(MPG_ERR_INVALID_ARG, "negative key_splits");
  if (d != 128) return fail(MPG_ERR_UNSUPPORTED, "head dimension %lld: only 128 is supported", (long long)d);
  if (lq == 0) return MPG_OK;
  if (lk == 0) return fail(MPG_ERR_INVALID_ARG, "softmax over zero keys");
  if (ldq < d || ldk < d || ldv < d || ldo < d)
    return fail(MPG_ERR_INVALID_ARG, "leading dimension smaller than d");
  if (!Q || !K || !V || !O) return fail(MPG_ERR_INVALID_ARG, "NULL operand");
  if (reinterpret_cast<uintptr_t>(Q) % 4 || reinterpret_cast<uintptr_t>(O) % 4)
    return fail(MPG_ERR_INVALID_ARG, "Q or O not aligned to 4 bytes");
  if (reinterpret_cast<uintptr_t>(K) % 16 || reinterpret_cast<uintptr_t>(V) % 16 || ldk % 8 || ldv % 8)
    return fail(MPG_ERR_INVALID_ARG, "K and V need 16-byte aligned pointers and leading dimensions (multiples of 8)");
  if (!std::isfinite(scale)) return fail(MPG_ERR_INVALID_ARG, "scale is not finite");
  DeviceInfo* dev = nullptr;
  mpg_status s = get_device(&dev);
  if (s != MPG_OK) return s;
  if (attention_smem_bytes() > dev->max_smem_optin)
    return fail(MPG_ERR_UNSUPPORTED, "attention kernel needs %d bytes of shared memory", attention_smem_bytes());
  AttnSplit sp = attention_split(lq, lk, key_splits, dev->sm_count);
  if (sp.splits > 1 && (!workspace || workspace_bytes < sp.bytes || reinterpret_cast<uintptr_t>(workspace) % 16)) {
    if (key_splits > 1)
      return fail(MPG_ERR_WORKSPACE, "%d key ranges need %zu workspace bytes (16-byte aligned), got %zu", sp.splits,
                  sp.bytes, workspace ? workspace_bytes : (size_t)0);
    sp = attention_split(lq, lk, 1, dev->sm_count);   // automatic choice: one range, no workspace
  }
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  Operand Kop{K, ldk, 0, MPG_F16, MPG_ROW_MAJOR};
  Operand Vop{V, ldv, 0, MPG_F16, MPG_ROW_MAJOR};
  s = encode_map(&p.map_k, Kop, d, lk, 1, 64, 64);
  if (s != MPG_OK) return s;
  s = encode_map(&p.map_v, Vop, d, lk, 1, 64, 64);
  if (s != MPG_OK) return s;
  p.q = Q;
  p.ldq = ldq;
  p.o = O;
  p.ldo = ldo;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.part_o = sp.splits > 1 ? reinterpret_cast<float*>(ws) : nullptr;
  p.part_m = sp.splits > 1 ? reinterpret_cast<float*>(ws + sp.off_m) : nullptr;
  p.part_l = sp.splits > 1 ? reinterpret_cast<float*>(ws + sp.off_l) : nullptr;
  p.lq = (int32_t)lq;
  p.lk = (int32_t)lk;
  p.splits = sp.splits;
  p.kb_per_split = sp.kb_per_split;
  p.num_q_blk = (int32_t)((lq + 127) / 128);
  p.q_vec_ok = (reinterpret_cast<uintptr_t>(Q) % 16 == 0) && (ldq % 4 == 0);
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.status = dev->status;
  p.wait_limit_ns = kDefaultWaitNs;
  if ((int64_t)p.num_q_blk * p.splits > 0x7FFFFFFF) return fail(MPG_ERR_INVALID_ARG, "too many CTAs");
  cudaError_t e = launch_attention(p, mode == MPG_ATTN_SPLIT_2CHAIN, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(MPG_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  return MPG_OK;
}

}  // extern "C"
