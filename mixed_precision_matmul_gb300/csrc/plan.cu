// Planning and launch of the tensor-core product: which kernel (path,
// conversion, tile width, CTA pairs), split-K, the separate conversion pass,
// aligned copies of operands TMA cannot describe, argument validation, and
// the launch with its tensor maps.  Nothing here allocates device memory.
#include <cmath>
#include <cstring>

#include "host.h"

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

// Tile width along N among widest, widest / 2, ... 64 (no wider than N
// needs): the least (rounds of tiles over the SMs) x (128 + width), a model
// of the time when every tile loads a 128-row A tile and a width-wide B tile
// per k-block; ties keep the wider tile.  Large products keep the widest
// tiles; products with fewer tiles than SMs take narrower, more numerous
// ones (256^3 fp16 on fp32 operands: 14 -> 7.5 us; 512^3 17 -> 11 us).
int pick_bn(int64_t m, int64_t n, int64_t batch, int splits, int sm_count, int widest) {
  int top = n <= 64 ? 64 : (n <= 128 ? std::min(widest, 128) : widest);
  int best = top;
  int64_t best_cost = -1;
  for (int w = top; w >= 64; w /= 2) {
    const int64_t tiles = batch * ((m + 127) / 128) * ((n + w - 1) / w) * std::max(splits, 1);
    const int64_t cost = ((tiles + sm_count - 1) / sm_count) * (128 + w);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = w;
    }
  }
  return best;
}

size_t tail_bytes(int64_t tiles) {
  return align256((size_t)tiles * 2 * 256 * 256 * sizeof(float)) + align256((size_t)tiles * 16 * sizeof(uint32_t));
}

// The library's choice of the split tail for `tiles` pair tiles on P
// clusters and num_k_blk k-blocks (64 elements, 32 for tf32).  Cutting the
// last round's tiles in two saves half a tile's time but pairs two
// clusters' halves: the second
// half waits for the later of the two (the clusters drift apart over the
// earlier rounds) and then exchanges 128 KB of partial sums per CTA, about
// 16 us in all on a GB300.  So: at least 128 k-blocks (k >= 8192 for 16-bit
// operands, 4096 for tf32: a tile takes about 50 us), at most 6 full rounds before the tail (more, and the
// one partial round is a small share of the time), and a last round of at
// most P / 2 tiles, so that every half finds a cluster.
bool tail_auto(int64_t tiles, int64_t P, int64_t num_k_blk) {
  const int64_t full = tiles / P, rem = tiles % P;
  return full >= 1 && full <= 6 && rem >= 1 && 2 * rem <= P && num_k_blk >= 128;
}

// The most split-tail workspace a call may take: at most a quarter of the
// SMs' worth of tiles by default (2R <= P <= SMs / 2 clusters), half with
// tail_split = 1; only the fp16 / bf16 / tf32 modes reach the pair kernel
// (k-blocks of 64 elements, 32 for tf32).
size_t tail_bound(int64_t m, int64_t n, int64_t k, int64_t batch, mpg_precision mode, int sm_count,
                  const mpg_options& o) {
  if (o.tail_split < 0 || (mode != MPG_FP16_F32ACC && mode != MPG_BF16_F32ACC && mode != MPG_TF32) ||
      o.cta_pair < 0)
    return 0;
  const int64_t bk = (mode == MPG_TF32) ? 32 : 64;
  if (o.tail_split == 1) return tail_bytes(std::max(sm_count / 2, 1));
  // the clusters resident at launch are at most SMs / 2, so a product this
  // query leaves out has more than 6 full rounds at launch too
  const int64_t P = std::max(sm_count / 2, 1);
  const int64_t pair_tiles = batch * ((m + 255) / 256) * ((n + 255) / 256);
  if (m <= 128 || n <= 128 || pair_tiles < P || pair_tiles / P > 6 || (k + bk - 1) / bk < 128) return 0;
  return tail_bytes(std::max(sm_count / 4, 1));
}

// Workspace of the separate conversion pass: packed 16-bit copies of A and B
// (hi and lo for the split) after the split-K partials, each 256-byte aligned.
// A copy keeps its operand's majorness; its lines are padded to a multiple of
// 8 elements so that every line starts on a 16-byte boundary (TMA).


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
  return c == Conv::kSplit3 || c == Conv::kSplit1 || c == Conv::kSplitA2 || c == Conv::kSplit4 ||
         c == Conv::kSplit3M;
}
bool splits_b(Conv c) {
  return c == Conv::kSplit3 || c == Conv::kSplit1 || c == Conv::kSplit4 || c == Conv::kSplit3M;
}

// Exponent L of the lo half's scale 2^L: 11 for the forms whose lo products
// have chains of their own, unless the caller asks for the plain lo; 0 for
// the one-chain form (and for conversions without a lo half).
int split_lo_exp(Conv c, const mpg_options& o) {
  if (c == Conv::kSplit3 || c == Conv::kSplitA2 || c == Conv::kSplit4 || c == Conv::kSplit3M)
    return o.split_plain_lo ? 0 : 11;
  return 0;
}

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
      // hi*lo and lo*hi in one shared accumulator when asked for and the
      // whole K range is one accumulation chunk
      p.conv = (o.split_lo_shared && (o.split_chunk_k < 0 ||
                                      k <= (o.split_chunk_k > 0 ? (int64_t)o.split_chunk_k : kDefaultSplitChunkK)))
                   ? Conv::kSplit3M
                   : Conv::kSplit3;
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
  size_t copies_end = 0;   // end of the conversion pass's or the aligned copies' region
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
      // a transposing copy runs on a grid of 32 x 32 blocks: batches and
      // blocks along the copy's lines within the grid's y and z limits
      auto transpose_fits = [&](bool copy, mpg_layout in, mpg_layout out, int64_t ld) {
        return !copy || in == out || (batch <= 65535 && (ld + 31) / 32 <= 65535);
      };
      if (L.end <= ws_bytes && transpose_fits(ca, A.layout, a_out, L.a_ld) &&
          transpose_fits(cb, B.layout, b_out, L.b_ld)) {
        p.src = Src::kTmaDirect;
        p.copy_a = ca;
        p.copy_b = cb;
        copies_end = L.end;
      }
    }
  }

  // tile width along N
  int bn;
  if (p.conv == Conv::kSplit4) {
    bn = 64;   // four chains of 64 columns plus the running sum fill TMEM
  } else if (p.src == Src::kGeneric) {
    bn = pick_bn(m, n, batch, splits, sm_count, 128);
  } else if (p.conv == Conv::kSplit3 || p.conv == Conv::kSplitA2 || p.conv == Conv::kSplit1 ||
             p.conv == Conv::kSplit3M) {
    // 128-wide tiles read A once per 128 columns; for the three-chain and
    // A-only splits they hold one TMEM accumulator, 64-wide tiles two
    bn = pick_bn(m, n, batch, splits, sm_count, 128);
  } else {
    // direct 16-bit / tf32, and fp32 -> fp16 / bf16 on load (the widest
    // tile converts the fewest source bytes per flop)
    bn = pick_bn(m, n, batch, splits, sm_count, 256);
  }
  if (o.tile_n != 0) {
    TcKernel probe;
    if (!tc_kernel_lookup(p.src, p.conv, p.op, p.st, o.tile_n, &probe))
      return fail(MPG_ERR_UNSUPPORTED, "tile_n %d is not available on this path", o.tile_n);
    bn = o.tile_n;
  }
  p.bn = bn;
  // CTA pairs: 16-bit or tf32 operands on the direct path (also the
  // conversion pass's and the aligned copies), 256 x 256 tiles.  Chosen by
  // the library when those tiles give every pair of SMs at least one and
  // the product is wider and taller than 128 (where the one-CTA kernel
  // would take 128 x 256 tiles too: narrower products, e.g. many small
  // batched ones, keep the finer tiles instead of multiplying padding), or
  // forced with cta_pair = 1.
  // The three-chain split on the conversion pass's copies also runs on
  // pairs, with 256 x 128 tiles, when asked for (cta_pair = 1).  Measured on
  // a GB300 at 4096^3 it is slower than single CTAs (360 against 412
  // TFLOP/s with 512-k chunks, 428 against 444 with one chunk), so the
  // library's own choice keeps single CTAs for the split.
  const bool split_pair = p.prepass && p.conv == Conv::kSplit3;
  const int pair_bn = split_pair ? 128 : 256;
  const bool pair_ok = p.src == Src::kTmaDirect && (p.conv == Conv::kNone || split_pair) &&
                       (o.tile_n == 0 || o.tile_n == pair_bn);
  const int64_t pair_tiles = batch * ((m + 255) / 256) * ((n + pair_bn - 1) / pair_bn);
  if (pair_ok && (o.cta_pair == 1 || (o.cta_pair == 0 && !split_pair && o.tile_n == 0 && m > 128 && n > 128 &&
                                      pair_tiles * 2 >= sm_count))) {
    p.pair = true;
    p.bn = pair_bn;
  }

  if (p.prepass) {
    const PrepassLayout L = prepass_layout(m, n, k, batch, A.layout, B.layout, splits_a(p.conv), splits_b(p.conv),
                                           splitk_bytes(splits, m, n, batch));
    if (L.end > ws_bytes)
      return fail(MPG_ERR_WORKSPACE, "the separate conversion pass needs %zu workspace bytes, got %zu", L.end,
                  ws_bytes);
    copies_end = L.end;
  }
  if (splits > 1 && splitk_bytes(splits, m, n, batch) > ws_bytes) {
    if (o.splitk > 0)
      return fail(MPG_ERR_WORKSPACE, "split-K with %d partitions needs %zu workspace bytes, got %zu", splits,
                  splitk_bytes(splits, m, n, batch), ws_bytes);
    splits = 1;  // automatic choice: no workspace, no split
  }
  p.splits = splits;
  // the split tail's partial sums follow everything else in the workspace
  p.tail_off = align256(std::max(copies_end, splitk_bytes(splits, m, n, batch)));
  p.tail_avail = ws_bytes > p.tail_off ? ws_bytes - p.tail_off : 0;
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
  // batches of C written concurrently must not share elements
  if (batch > 1 && strideC > 0 && m > 0 && n > 0 && strideC < (m - 1) * ldc + n)
    return fail(MPG_ERR_INVALID_ARG, "strideC=%lld makes the batch matrices of C overlap (one spans %lld elements)",
                (long long)strideC, (long long)((m - 1) * ldc + n));
  if (o.split_exp_a < -100 || o.split_exp_a > 100 || o.split_exp_b < -100 || o.split_exp_b > 100)
    return fail(MPG_ERR_INVALID_ARG, "split exponent outside [-100, 100]");
  if (o.splitk < 0) return fail(MPG_ERR_INVALID_ARG, "negative splitk");
  if (o.wait_timeout_ns < 0) return fail(MPG_ERR_INVALID_ARG, "negative wait timeout");
  if (o.c_dtype < MPG_F32 || o.c_dtype > MPG_BF16) return fail(MPG_ERR_INVALID_ARG, "unknown C dtype %d", o.c_dtype);
  if (o.cta_pair < -1 || o.cta_pair > 1) return fail(MPG_ERR_INVALID_ARG, "cta_pair must be -1, 0 or 1");
  if (o.tail_split < -1 || o.tail_split > 1) return fail(MPG_ERR_INVALID_ARG, "tail_split must be -1, 0 or 1");
  if (o.prepass < -1 || o.prepass > 1) return fail(MPG_ERR_INVALID_ARG, "prepass must be -1, 0 or 1");
  if (o.split_plain_lo < 0 || o.split_plain_lo > 1)
    return fail(MPG_ERR_INVALID_ARG, "split_plain_lo must be 0 or 1");
  if (o.split_lo_shared < 0 || o.split_lo_shared > 1)
    return fail(MPG_ERR_INVALID_ARG, "split_lo_shared must be 0 or 1");
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

// Clusters of two CTAs of a pair kernel that fit on the device at once,
// asked once per device and launch shape (the plain pair kernels share one;
// the split's has less shared memory).
mpg_status pair_clusters(DeviceInfo* dev, const TcKernel& kern, int* out) {
  static std::mutex mu;
  static int cached[kMaxDevices][2];
  const int devid = (int)(dev - g_devices);
  const int shape = kern.bn == 128 ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  int& slot = cached[devid][shape];
  if (slot <= 0) {
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
    slot = n;
  }
  *out = slot;
  return MPG_OK;
}

mpg_status launch_tc(const Plan& plan, DeviceInfo* dev, int64_t m, int64_t n, int64_t k, int64_t batch,
                     const Operand& A, const Operand& B, float* C, int64_t ldc, int64_t strideC, float alpha,
                     float beta, const mpg_options& o, void* workspace, cudaStream_t stream,
                     const Operand* A_lo, const Operand* B_lo, bool dependent) {
  TcKernel kern;
  const bool found = plan.pair ? mpg::tc_lookup_pair(plan.op, plan.conv, &kern)
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
  p.tail_first = p.num_tiles;
  // clusters of the pair kernel resident at once
  int clusters = 0;
  if (plan.pair) {
    mpg_status cs = pair_clusters(dev, kern, &clusters);
    if (cs != MPG_OK) return cs;
  }
  // split tail: the last round's R tiles become 2R halves of their k range
  int64_t tail_tiles = 0;
  if (plan.pair && plan.conv == Conv::kNone && splits_eff == 1 && o.tail_split >= 0 && p.num_k_blk >= 2 &&
      tiles > 0) {
    const int64_t P = clusters;
    const int64_t full = tiles / P, rem = tiles % P;
    if (o.tail_split == 1) {
      tail_tiles = full == 0 ? tiles : rem;
    } else if (tail_auto(tiles, P, p.num_k_blk) && tail_bytes(rem) <= plan.tail_avail) {
      tail_tiles = rem;
    }
    if (tail_tiles > 0 && tail_bytes(tail_tiles) > plan.tail_avail)
      return fail(MPG_ERR_WORKSPACE, "the split tail needs %zu workspace bytes after offset %zu, got %zu",
                  tail_bytes(tail_tiles), plan.tail_off, plan.tail_avail);
  }
  if (tail_tiles > 0) {
    uint8_t* base = static_cast<uint8_t*>(workspace) + plan.tail_off;
    p.tail_first = (int32_t)(tiles - tail_tiles);
    p.num_tiles = (int32_t)(tiles + tail_tiles);
    p.tail_kb_mid = p.num_k_blk / 2;
    p.tail_ws = reinterpret_cast<float*>(base);
    p.tail_cnt = reinterpret_cast<uint32_t*>(base + align256((size_t)tail_tiles * 2 * 256 * 256 * sizeof(float)));
    cudaError_t me = cudaMemsetAsync(p.tail_cnt, 0, (size_t)tail_tiles * 16 * sizeof(uint32_t), stream);
    if (me != cudaSuccess) return fail(MPG_ERR_CUDA, "split tail counters: %s", cudaGetErrorString(me));
  }
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
  // TMA stores of the one-CTA epilogue: fp32 results without a C to read
  // (beta == 0) on 16-byte aligned lines, or the split-K partial sums.
  // Only when a row of the result is a whole number of 16-byte chunks
  // (n % 4 == 0): measured on a GB300, a store box that ends inside a
  // 16-byte chunk of a row wrote the rest of that chunk (C's padding).
  p.tma_store = 0;
  if (!plan.pair && n % 4 == 0) {
    mpg_status ms = MPG_OK;
    if (splits_eff > 1 && p.p_vec_ok) {
      const Operand P{workspace, n, m * n, MPG_F32, MPG_ROW_MAJOR};
      ms = encode_map(&p.map_out, P, n, m, (int64_t)splits_eff * batch, 32, 32);
      p.tma_store = 1;
    } else if (splits_eff == 1 && beta == 0.0f && o.c_dtype == MPG_F32 && p.c_vec_ok) {
      const Operand Cop{C, ldc, p.stride_c, MPG_F32, MPG_ROW_MAJOR};
      if (tma_ok(Cop, batch)) {
        ms = encode_map(&p.map_out, Cop, n, m, batch, 32, 32);
        p.tma_store = 1;
      }
    }
    if (ms != MPG_OK) return ms;
  }
  const bool split = splits_a(plan.conv);
  const int sa = split ? o.split_exp_a : 0, sb = split ? o.split_exp_b : 0;
  p.alpha = (float)std::ldexp((double)alpha, -(sa + sb));
  p.beta = beta;
  p.scale_a = std::ldexp(1.0f, sa);
  p.scale_b = std::ldexp(1.0f, sb);
  const int lo_exp = split_lo_exp(plan.conv, o);
  p.lo_mul = std::ldexp(1.0f, lo_exp);
  p.lo_inv = std::ldexp(1.0f, -lo_exp);
  p.status = dev->status;
  p.wait_limit_ns = o.wait_timeout_ns > 0 ? (uint64_t)o.wait_timeout_ns : kDefaultWaitNs;
  p.chunk_kb = 0;
  // K chunks of the split's accumulation: the default for the three- and
  // four-chain splits; the A-only split takes one chunk by default (its
  // error is set by B's fp16 rounding, 100x the tensor cores' accumulation
  // error over the whole K), any of them the caller's chunk when given
  const bool chunked = (plan.conv == Conv::kSplit3 || plan.conv == Conv::kSplit4) ? o.split_chunk_k >= 0
                       : plan.conv == Conv::kSplitA2                             ? o.split_chunk_k > 0
                                                                                 : false;
  if (chunked) {
    const int64_t chunk_k = o.split_chunk_k > 0 ? o.split_chunk_k : kDefaultSplitChunkK;
    p.chunk_kb = (int32_t)std::min<int64_t>((chunk_k + BK - 1) / BK, p.num_k_blk);
  }

  void* args[] = {&p};
  cudaError_t e;
  {
    // persistent grid: clusters of two CTAs for the pair kernels (as many
    // clusters as can be resident at once), one CTA per SM otherwise.  A
    // product whose operands the previous kernel of this call wrote (the
    // conversion pass, aligned copies) is that kernel's programmatic
    // dependent: its set-up overlaps the other's end (the kernel waits with
    // griddepcontrol.wait before reading anything).
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = plan.pair ? dim3((unsigned)(2 * std::min<int64_t>(p.num_tiles, clusters)))
                            : dim3((unsigned)std::min<int64_t>(tiles, dev->sm_count));
    cfg.blockDim = dim3((unsigned)kern.block);
    cfg.dynamicSmemBytes = (size_t)kern.smem_bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (plan.pair) {
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = 2;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = 1;
      ++na;
    }
    if (dependent) {
      attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[na].val.programmaticStreamSerializationAllowed = 1;
      ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    e = cudaLaunchKernelExC(&cfg, kern.fn, args);
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

}  // namespace mpg
