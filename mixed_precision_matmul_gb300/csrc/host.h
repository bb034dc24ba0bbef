// Host-side internals shared by the translation units of the C ABI:
// error reporting, the per-device cache, operand descriptions, the plan of a
// product (kernel, tile width, split-K, conversion pass, aligned copies) and
// its launch.  Not part of the public interface (include/mpgemm.h is).
#pragma once

#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <string>

#include "internal.h"
#include "mpgemm.h"

namespace mpg {

// ---- errors: the thread's last message (mpg_last_error_string)
extern thread_local std::string t_err;
mpg_status fail(mpg_status s, const char* fmt, ...);

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
// K chunk of the three- and four-chain splits' accumulation: measured on
// the log-uniform 4096^3 product, error vs FFMA 0.25x / 0.45x / 0.66x / 1.33x
// for chunks of 256 / 512 / 1024 / 2048, speed 361 / 408 / 431 / 445 TFLOP/s.
constexpr int64_t kDefaultSplitChunkK = 512;


struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int max_smem_optin = 0;
  uint32_t* status = nullptr;
  std::atomic<uint64_t> smem_set_mask[4];  // kernels whose smem attribute was set (by slot)
};

extern DeviceInfo g_devices[kMaxDevices];

// The cached description of the current device (checked to be sm_103).
mpg_status get_device(DeviceInfo** out);

inline int elem_bytes(mpg_dtype t) { return t == MPG_F32 ? 4 : 2; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ---- plans
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
  size_t tail_off = 0;        // workspace offset of the split tail's partial sums and counters
  size_t tail_avail = 0;      // workspace bytes from tail_off on
};

struct Operand {
  const void* ptr;
  int64_t ld, stride;
  mpg_dtype dt;
  mpg_layout layout;
};

// TMA can describe the operand (16-byte aligned base, leading dimension and
// batch stride).
bool tma_ok(const Operand& x, int64_t batch);
void resolve_options(const mpg_options* opt, mpg_options* o);
// 3-D map {inner, outer, batch}, box {box_inner, box_outer, 1}, 128B swizzle.
mpg_status encode_map(CUtensorMap* map, const Operand& x, int64_t inner, int64_t outer, int64_t batch,
                      int box_inner, int box_outer);

int choose_splits(int64_t m, int64_t n, int64_t k, int64_t batch, int sm_count, const mpg_options& o);
size_t splitk_bytes(int splits, int64_t m, int64_t n, int64_t batch);
// Workspace of the CTA-pair kernel's split tail for `tiles` tiles: two
// halves of fp32 partial sums per 256 x 256 tile, then one counter per
// epilogue warp piece; and its bound for the workspace queries.
size_t tail_bytes(int64_t tiles);
int pick_bn(int64_t m, int64_t n, int64_t batch, int splits, int sm_count, int widest);
size_t tail_bound(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_precision mode, int sm_count,
                  const mpg_options& o);
bool tail_auto(int64_t tiles, int64_t clusters, int64_t num_k_blk);
struct PrepassLayout {
  int64_t a_outer, a_inner, a_ld, b_outer, b_inner, b_ld;
  size_t off_a_hi, off_a_lo, off_b_hi, off_b_lo, end;
};
PrepassLayout prepass_layout(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_layout al, mpg_layout bl,
                             bool split_a, bool split_b, size_t base);
struct CopyLayout {
  mpg_layout a_layout, b_layout;                 // layouts of the copies
  int64_t a_outer, a_inner, a_ld, b_outer, b_inner, b_ld;
  size_t off_a, off_b, end;
};
CopyLayout copy_layout(int64_t m, int64_t n, int64_t k, int64_t batch, const Operand& A, const Operand& B,
                       bool ca, bool cb, size_t base, mpg_layout a_out, mpg_layout b_out);
bool split_mode(mpg_precision mode);
bool auto_prepass_shape(int64_t m, int64_t n, int64_t k);
bool prepass_mode(mpg_precision mode);
bool splits_a(Conv c);
bool splits_b(Conv c);
int split_lo_exp(Conv c, const mpg_options& o);
mpg_status make_plan(int64_t m, int64_t n, int64_t k, int64_t batch, const Operand& A, const Operand& B,
                     float alpha, mpg_precision mode, const mpg_options& o, int sm_count, size_t ws_bytes,
                     Plan* plan);
mpg_status validate(int64_t m, int64_t n, int64_t k, int64_t batch, const Operand& A, const Operand& B,
                    const float* C, int64_t ldc, int64_t strideC, float alpha, mpg_precision mode,
                    const mpg_options& o);
mpg_status launch_tc(const Plan& plan, DeviceInfo* dev, int64_t m, int64_t n, int64_t k, int64_t batch,
                     const Operand& A, const Operand& B, float* C, int64_t ldc, int64_t strideC, float alpha,
                     float beta, const mpg_options& o, void* workspace, cudaStream_t stream,
                     const Operand* A_lo = nullptr, const Operand* B_lo = nullptr, bool dependent = false);

}  // namespace mpg
