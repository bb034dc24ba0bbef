// The tensor-core product C = alpha*A*B + beta*C for sm_103a.
//
// One persistent, warp-specialised kernel template:
//   warp 0       TMA producer (direct and staged paths)
//   warp 1       TMEM allocator and the single thread that issues tcgen05.mma
//   warps 2..    epilogue: tcgen05.ld -> chain sum -> alpha/beta -> stores
//                (4 warps, one per TMEM lane quarter; 8 on the direct path,
//                two per quarter, each taking half of the tile's columns)
//   then         converters (staged and generic paths, 8 warps): fp32 ->
//                fp16/bf16 or the hi/lo split, written into the swizzled
//                operand stages
//
// The accumulator lives in TMEM for the whole K loop (the register/accumulator
// residency of "tile_matmul(): use the cuBLASDx register-accumulator API ...",
// "Proposed change"); operand stages use the 128-byte (64-byte for 64-byte
// lines) swizzled layouts so the tensor core reads them without bank
// conflicts ("... suggested (swizzled) shared layouts").  The hi/lo chains of
// the split modes follow "qsa_prompt_attn: ... keep the hi and lo halves in
// separate accumulator chains", section "The fix".
//
// Accumulator layout (M = 128, cta_group::1): row i of the tile is TMEM lane i,
// column j is TMEM column (buffer base + j).  Warp w reads lanes 32*(w%4) ..
// 32*(w%4)+31 with tcgen05.ld.32x32b.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "outio.cuh"
#include "ptx.cuh"
#include "staging.cuh"

namespace mpg {

template <Src S, Conv CV, Op O, SrcT ST, int BN_>
struct TcTraits {
  static constexpr Src kSrc = S;
  static constexpr Conv kConv = CV;
  static constexpr Op kOp = O;
  static constexpr SrcT kSrcT = ST;
  static constexpr int BM = 128;
  static constexpr int BN = BN_;
  static constexpr int kOpBytes = (O == Op::kTF32) ? 4 : 2;
  // k elements per stage: 128-byte lines for the direct path, 32 elements
  // (one 128-byte line of fp32 source) for the converter paths.
  static constexpr int BK = (S == Src::kTmaDirect) ? (128 / kOpBytes) : 32;
  static constexpr int kRowBytes = BK * kOpBytes;  // 128 or 64
  static constexpr uint32_t kSwizzle = (kRowBytes == 128) ? kSwizzle128B : kSwizzle64B;
  static constexpr int kKSteps = kRowBytes / 32;   // MMAs of 32 bytes of K each
  static constexpr int kInstrK = 32 / kOpBytes;    // 16 (f16/bf16) or 8 (tf32)
  // operands that carry a hi and a lo copy in the stages
  static constexpr bool kSplitA = (CV == Conv::kSplit3 || CV == Conv::kSplit1 || CV == Conv::kSplitA2 ||
                                    CV == Conv::kSplit4 || CV == Conv::kSplit3M);
  static constexpr bool kSplitB =
      (CV == Conv::kSplit3 || CV == Conv::kSplit1 || CV == Conv::kSplit4 || CV == Conv::kSplit3M);
  static constexpr int kCopiesA = kSplitA ? 2 : 1;
  static constexpr int kCopiesB = kSplitB ? 2 : 1;
  static constexpr int kATile = BM * kRowBytes;
  static constexpr int kBTile = BN * kRowBytes;
  static constexpr int kOpStage = kCopiesA * kATile + kCopiesB * kBTile;
  static constexpr bool kStaged = (S == Src::kTmaStaged);
  static constexpr bool kHasConv = (S != Src::kTmaDirect);
  static constexpr int kStgATile = kStaged ? BM * 128 : 0;
  static constexpr int kStgBTile = kStaged ? BN * 128 : 0;
  static constexpr int kStgStage = kStgATile + kStgBTile;
  static constexpr int kBudget = 196 * 1024;
  // Ring depths.  Without staging one ring of operand stages carries the
  // loads in flight.  On the staged path the fp32 staging ring (TMA from L2
  // or HBM) carries them and the ring of converted operand stages the
  // hand-off from the converter warps to the MMAs: equal depths where the
  // budget gives both three or more stages (measured best for the splits),
  // else two operand stages and the rest to staging (fp32 -> fp16 / bf16 on
  // 256-wide tiles: 2 + 3 stages instead of 2 + 2, 443 -> 529 TFLOP/s at
  // 8192^3; two operand stages with the splits' larger ones measured slower).
  static constexpr int kEqualRaw = kBudget / (kOpStage + kStgStage);
  static constexpr int kEqual = kEqualRaw > 8 ? 8 : kEqualRaw;
  static constexpr int kOpRaw = !kStaged ? kBudget / kOpStage : (kEqual >= 3 ? kEqual : 2);
  static constexpr int kStagesOp = kOpRaw > 8 ? 8 : kOpRaw;
  static constexpr int kStgRaw =
      !kStaged ? 0 : (kEqual >= 3 ? kEqual : (kBudget - kStagesOp * kOpStage) / kStgStage);
  static constexpr int kStagesStg = kStgRaw > 8 ? 8 : kStgRaw;
  static_assert(kStagesOp >= 2 && (!kStaged || kStagesStg >= 2), "pipeline needs two stages");
  static constexpr int kConvWarps = kHasConv ? 8 : 0;
  static constexpr int kConvThreads = kConvWarps * 32;
  static constexpr int kEpiWarps = kHasConv ? 4 : 8;
  static constexpr int kEpiThreads = kEpiWarps * 32;
  static constexpr int kConvWarp0 = 2 + kEpiWarps;    // first converter warp
  static constexpr int kThreads = (2 + kEpiWarps + kConvWarps) * 32;
  // TMEM: columns of one accumulator (all chains), buffers, allocation.
  // The three-chain split accumulates K in chunks: each chunk starts fresh
  // chains, and the epilogue folds hh + 2^-11 (hl + lh) of every chunk into
  // an fp32 running sum (round to nearest) kept in kRunCols extra columns.
  static constexpr bool kPromote = (CV == Conv::kSplit3 || CV == Conv::kSplitA2 || CV == Conv::kSplit4);
  // The two-accumulator split (hh; hl + lh) covers one K chunk and needs no
  // running sum, so two of its accumulators fit in TMEM: the epilogue of one
  // tile overlaps the MMAs of the next.
  static constexpr int kChainCols = (CV == Conv::kSplit4)                            ? 4 * BN
                                    : (CV == Conv::kSplit3)                           ? 3 * BN
                                    : (CV == Conv::kSplitA2 || CV == Conv::kSplit3M) ? 2 * BN
                                                                                      : BN;
  static constexpr int kRunCols = kPromote ? BN : 0;
  static constexpr int kAccStride = kPromote ? kChainCols
                                    : kChainCols <= 32 ? 32 : kChainCols <= 64 ? 64 : kChainCols <= 128 ? 128
                                    : kChainCols <= 256 ? 256 : 512;
  static constexpr int kAccBufs = (2 * kAccStride + kRunCols <= 512) ? 2 : 1;
  static constexpr int kRunBase = kAccBufs * kAccStride;
  static constexpr int kTmemUsed = kRunBase + kRunCols;
  static constexpr int kTmemCols = kTmemUsed <= 32 ? 32 : kTmemUsed <= 64 ? 64 : kTmemUsed <= 128 ? 128
                                   : kTmemUsed <= 256 ? 256 : 512;
  static_assert(kTmemUsed <= 512, "TMEM budget");
  static constexpr int kEpiBytes = kEpiWarps * 32 * 32 * 4;
  static constexpr int kNumBars = 2 * kStagesOp + 2 * kStagesStg + 2 * kAccBufs + 1;
  static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStagesOp * kOpStage + kStagesStg * kStgStage + kEpiBytes +
                                    kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // each epilogue warp's staging buffer starts on a 1024-byte boundary (the
  // 128-byte swizzle of its TMA stores repeats every 1024 bytes)
  static_assert((kStagesOp * kOpStage) % 1024 == 0 && (kStagesStg * kStgStage) % 1024 == 0, "staging alignment");
  static_assert(BN % BK == 0 && BM % BK == 0, "regions of MN-major tiles");
  static constexpr uint32_t kAbFormat = (O == Op::kF16) ? 0u : (O == Op::kBF16) ? 1u : 2u;
};

struct TileCoord {
  int s, b, mb, nb, kb0, kb1;
  int tail;   // index among the tiles whose k range is cut in two, or -1
  int half;   // which half of the k range (0: [kb0, mid), 1: [mid, kb1))
};

__device__ __forceinline__ TileCoord decode_tile(const TcParams& p, int t) {
  TileCoord c;
  const int per_batch = p.num_m_blk * p.num_n_blk;
  const int per_split = per_batch * p.batch;
  c.s = t / per_split;
  int r = t - c.s * per_split;
  c.b = r / per_batch;
  r -= c.b * per_batch;
  const int G = p.group_m;
  const int group_size = G * p.num_n_blk;
  const int g = r / group_size;
  const int first_m = g * G;
  const int gm = min(G, p.num_m_blk - first_m);
  const int within = r - g * group_size;
  c.mb = first_m + within % gm;
  c.nb = within / gm;
  // serpentine: odd groups walk the columns backwards, starting on the B
  // panels the previous group read last (still in L2)
  if (g & 1) c.nb = p.num_n_blk - 1 - c.nb;
  c.kb0 = c.s * p.kb_per_split;
  c.kb1 = min(p.num_k_blk, c.kb0 + p.kb_per_split);
  c.tail = -1;
  c.half = 0;
  return c;
}

// Work item t of a persistent loop.  Items below tail_first are whole tiles
// in decode_tile's order; from tail_first on, each remaining tile is two
// items, the halves of its k range, so that the last round of tiles spreads
// over twice as many workers.
__device__ __forceinline__ TileCoord decode_item(const TcParams& p, int t) {
  if (t < p.tail_first) return decode_tile(p, t);
  const int h = t - p.tail_first;
  TileCoord c = decode_tile(p, p.tail_first + (h >> 1));
  c.tail = h >> 1;
  c.half = h & 1;
  if (c.half == 0) c.kb1 = p.tail_kb_mid;
  else c.kb0 = p.tail_kb_mid;
  return c;
}

// All lanes of the warp wait; the warp continues only if every lane succeeded.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& ctl) {
  const bool ok = mbar_wait(bar, parity, ctl);
  return __all_sync(0xffffffffu, ok);
}

// Waits used at teardown: bounded, but independent of the abort flag, so that
// copies and MMAs already in flight finish before the CTA releases its
// shared memory and TMEM.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test(bar, parity)) return;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 30); ++it) {
    if (mbar_test(bar, parity)) return;
    if ((it & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return;
  }
}

// Byte offset of 16-byte chunk `ch` of line `line` in a swizzled tile whose
// lines are `RB` bytes: 128B pattern XORs chunk bits [4,7) with address bits
// [7,10); the 64B pattern XORs bits [4,6) with bits [7,9).
template <int RB>
__device__ __forceinline__ uint32_t swz_chunk_offset(uint32_t line, uint32_t ch) {
  if constexpr (RB == 128) {
    return line * 128u + ((ch ^ (line & 7u)) << 4);
  } else {
    return line * 64u + ((ch ^ ((line >> 1) & 3u)) << 4);
  }
}

template <class T>
__device__ __forceinline__ uint64_t operand_desc(uint32_t tile_addr, bool mn_major, int ks) {
  constexpr uint32_t RB = T::kRowBytes;
  if (!mn_major) {
    // K-major: 8-line swizzle atoms stacked along M/N at SBO = 8 lines; the
    // K step moves the start address by 32 bytes inside the 128/64-byte line.
    return make_smem_desc(tile_addr + ks * 32u, 16u, 8u * RB, T::kSwizzle);
  } else {
    // MN-major: atoms of (RB bytes of M/N) x (8 k-lines); regions of BK lines
    // repeat along M/N at LBO, 8-line groups along K at SBO.
    return make_smem_desc(tile_addr + ks * (uint32_t)T::kInstrK * RB, (uint32_t)T::BK * RB, 8u * RB, T::kSwizzle);
  }
}

// -------------------------------------------------------------------------
// converter helpers
// -------------------------------------------------------------------------
template <SrcT ST>
struct SrcElem;
template <>
struct SrcElem<SrcT::kF32> {
  using type = float;
  __device__ static float load(const float* p) { return __ldg(p); }
};
template <>
struct SrcElem<SrcT::kF16> {
  using type = unsigned short;
  __device__ static unsigned short load(const unsigned short* p) { return __ldg(p); }
};
template <>
struct SrcElem<SrcT::kBF16> {
  using type = unsigned short;
  __device__ static unsigned short load(const unsigned short* p) { return __ldg(p); }
};

__device__ __forceinline__ uint32_t pack_f16x2(float lo_elem, float hi_elem) {
  __half2 h = __floats2half2_rn(lo_elem, hi_elem);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo_elem, float hi_elem) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo_elem, hi_elem);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Split of two fp32 values: hi = fp16(x*s), lo = fp16((x*s - hi) * lo_mul),
// lo_mul = 2^L (1 or 2^11).  x*s and the residual are exact in fp32
// (power-of-two scale; the residual of an 11-bit rounding of a 24-bit
// significand has at most 13 bits), and so is the product with lo_mul.
__device__ __forceinline__ void split_pair(float x0, float x1, float s, float lo_mul, uint32_t& hi, uint32_t& lo) {
  const float y0 = x0 * s, y1 = x1 * s;
  __half2 h = __floats2half2_rn(y0, y1);
  const float2 hb = __half22float2(h);
  const float r0 = y0 - hb.x, r1 = y1 - hb.y;
  __half2 l = __floats2half2_rn(r0 * lo_mul, r1 * lo_mul);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
  asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}

// Convert 4 consecutive source values (fp32, or raw 16-bit codes) into the
// 32-bit words the operand tiles hold: for 16-bit operands w[0..1] are the
// four converted values (hi for the split) and w[2..3] the split's lo; for
// tf32 operands w[0..3] are the fp32 bits.
template <class T>
__device__ __forceinline__ void pack_chunk(const float (&x)[4], const unsigned short (&h)[4], float scale,
                                           float lo_mul, uint32_t (&w)[4], bool isA) {
  if constexpr (T::kOpBytes == 4) {
#pragma unroll
    for (int e = 0; e < 4; ++e) w[e] = __float_as_uint(x[e]);
  } else if constexpr (T::kConv == Conv::kNone) {
    w[0] = (uint32_t)h[0] | ((uint32_t)h[1] << 16);
    w[1] = (uint32_t)h[2] | ((uint32_t)h[3] << 16);
    w[2] = w[3] = 0;
  } else if constexpr (T::kConv == Conv::kRoundF16) {
    w[0] = pack_f16x2(x[0], x[1]);
    w[1] = pack_f16x2(x[2], x[3]);
    w[2] = w[3] = 0;
  } else if constexpr (T::kConv == Conv::kRoundBF16) {
    w[0] = pack_bf16x2(x[0], x[1]);
    w[1] = pack_bf16x2(x[2], x[3]);
    w[2] = w[3] = 0;
  } else if constexpr (T::kConv == Conv::kSplitA2) {
    // A is split (lo scaled by 2^11), B rounded to fp16
    if (isA) {
      split_pair(x[0], x[1], scale, lo_mul, w[0], w[2]);
      split_pair(x[2], x[3], scale, lo_mul, w[1], w[3]);
    } else {
      w[0] = pack_f16x2(x[0] * scale, x[1] * scale);
      w[1] = pack_f16x2(x[2] * scale, x[3] * scale);
      w[2] = w[3] = 0;
    }
  } else {
    split_pair(x[0], x[1], scale, lo_mul, w[0], w[2]);
    split_pair(x[2], x[3], scale, lo_mul, w[1], w[3]);
  }
}

// Store one packed chunk (line `lg`, 16-byte source chunk `ch`) into the
// operand tile(s) at `hi_tile` (and `lo_tile` for the split).
template <class T>
__device__ __forceinline__ void store_chunk(const uint32_t (&w)[4], uint32_t hi_tile, uint32_t lo_tile, uint32_t lg,
                                            uint32_t ch, bool transpose, bool isA) {
  if constexpr (T::kOpBytes == 4) {
    if (transpose) {
      // tf32 operands are kept K-major in shared memory: an MN-major source
      // chunk (k line `lg % BK`, 4 consecutive M/N values) scatters into 4
      // lines of the K-major tile
      const uint32_t kline = lg % T::BK;
      const uint32_t mn0 = (lg / T::BK) * T::BK + ch * 4;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t addr = hi_tile + swz_chunk_offset<128>(mn0 + e, kline >> 2) + ((kline & 3u) << 2);
        asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(w[e]) : "memory");
      }
    } else {
      // tf32 operand: fp32 copied into 128-byte swizzled lines
      st_shared_v4(hi_tile + swz_chunk_offset<128>(lg, ch), w[0], w[1], w[2], w[3]);
    }
  } else {
    // 16-bit operand, 64-byte lines: 4 values = half of a 16-byte chunk
    const uint32_t off = swz_chunk_offset<64>(lg, ch >> 1) + ((ch & 1u) << 3);
    st_shared_v2(hi_tile + off, w[0], w[1]);
    if ((isA && T::kSplitA) || (!isA && T::kSplitB)) st_shared_v2(lo_tile + off, w[2], w[3]);
  }
}

// -------------------------------------------------------------------------
// the kernel
// -------------------------------------------------------------------------
template <class T>
__global__ void __launch_bounds__(T::kThreads, 1) tc_gemm_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte aligned base (swizzle atoms repeat every 1024 bytes)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* op_base = smem;
  uint8_t* stg_base = op_base + T::kStagesOp * T::kOpStage;
  float* epi_base = reinterpret_cast<float*>(stg_base + T::kStagesStg * T::kStgStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(epi_base) + T::kEpiBytes);
  uint64_t* op_full = bars;                       // operand stage ready for the MMA
  uint64_t* op_empty = bars + T::kStagesOp;       // operand stage consumed by the MMA
  uint64_t* stg_full = bars + 2 * T::kStagesOp;   // staging filled by TMA
  uint64_t* stg_empty = stg_full + T::kStagesStg; // staging read by the converters
  uint64_t* acc_full = stg_empty + T::kStagesStg; // accumulator complete
  uint64_t* acc_empty = acc_full + T::kAccBufs;   // accumulator drained by the epilogue
  uint64_t* done_bar = acc_empty + T::kAccBufs;   // all MMAs of this CTA finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < T::kStagesOp; ++i) {
      if constexpr (T::kHasConv) {
        mbar_init(&op_full[i], T::kConvThreads);
      } else {
        mbar_init(&op_full[i], 1);
      }
      mbar_init(&op_empty[i], 1);
    }
    for (int i = 0; i < T::kStagesStg; ++i) {
      mbar_init(&stg_full[i], 1);
      mbar_init(&stg_empty[i], T::kConvThreads);
    }
    for (int i = 0; i < T::kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], T::kEpiThreads);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, T::kTmemCols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up above may overlap the end of the kernel that wrote this
  // product's operands (the conversion pass or aligned copies); nothing of
  // theirs is read before this point
  griddep_wait();
  griddep_launch_dependents();

  WaitCtl ctl;
  ctl.abort = abort_flag;
  ctl.status = p.status;
  ctl.limit_ns = p.wait_limit_ns;

  const uint32_t op_smem = smem_addr(op_base);
  const uint32_t stg_smem = smem_addr(stg_base);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if constexpr (T::kSrc != Src::kGeneric) {
      if (lane == 0) {
        tma_prefetch_map(&p.map_a);
        tma_prefetch_map(&p.map_b);
        // direct path: TMA into the operand stage (op_full/op_empty);
        // staged path: TMA into the staging buffer (stg_full/stg_empty)
        uint64_t* fullb = T::kStaged ? stg_full : op_full;
        uint64_t* emptyb = T::kStaged ? stg_empty : op_empty;
        constexpr int kLineBytes = T::kStaged ? 128 : T::kRowBytes;
        constexpr int kABytes = T::BM * kLineBytes;
        constexpr int kStageBytes = T::kStaged ? T::kStgStage : T::kOpStage;
        constexpr int kRegion = T::BK * kLineBytes;  // bytes of one MN-major region
        constexpr uint32_t kRing = T::kStaged ? T::kStagesStg : T::kStagesOp;   // the ring it fills
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
          const TileCoord tc = decode_tile(p, t);
          for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++it) {
            const uint32_t st = it % kRing;
            const uint32_t ph = (it / kRing) & 1u;
            if (!mbar_wait(&emptyb[st], ph ^ 1u, ctl)) { ok = false; break; }
            uint8_t* dst = (T::kStaged ? stg_base + st * T::kStgStage : op_base + st * T::kOpStage);
            mbar_arrive_expect_tx(&fullb[st], kStageBytes);
            const int k0 = kb * T::BK;
            // one operand tile: a single K-major box, or MN-major regions of BK
            auto load_tile = [&](const CUtensorMap* map, uint8_t* d, bool mn, int row0, int rows) {
              if (!mn) {
                tma_load_3d(d, map, &fullb[st], k0, row0, tc.b);
              } else {
                for (int g = 0; g < rows / T::BK; ++g)
                  tma_load_3d(d + g * kRegion, map, &fullb[st], row0 + g * T::BK, k0, tc.b);
              }
            };
            load_tile(&p.map_a, dst, p.a_mn_major, tc.mb * T::BM, T::BM);
            if constexpr (T::kSplitA && !T::kHasConv) {
              // pre-split operands: hi and lo halves of A, then of B (B may be single)
              load_tile(&p.map_a_lo, dst + T::kATile, p.a_mn_major, tc.mb * T::BM, T::BM);
              load_tile(&p.map_b, dst + 2 * T::kATile, p.b_mn_major, tc.nb * T::BN, T::BN);
              if constexpr (T::kSplitB)
                load_tile(&p.map_b_lo, dst + 2 * T::kATile + T::kBTile, p.b_mn_major, tc.nb * T::BN, T::BN);
            } else {
              load_tile(&p.map_b, dst + kABytes, p.b_mn_major, tc.nb * T::BN, T::BN);
            }
          }
        }
        // let copies already issued land before the CTA may exit
        const uint32_t n_drain = it < kRing ? it : kRing;
        for (uint32_t i = it - n_drain; i < it; ++i)
          drain_wait(&fullb[i % kRing], (i / kRing) & 1u, p.wait_limit_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // shared-memory majorness of the operands: 16-bit tiles keep the
      // source's majorness; tf32 tiles are always K-major
      const bool a_mn = (T::kOp == Op::kTF32) ? false : (p.a_mn_major != 0);
      const bool b_mn = (T::kOp == Op::kTF32) ? false : (p.b_mn_major != 0);
      uint32_t it = 0, g = 0;   // k-block iteration; accumulation chunk
      bool ok = true;
      const uint32_t idesc_n = make_idesc(T::kAbFormat, a_mn, b_mn, T::BM, T::BN);
      const uint32_t idesc_2n =
          make_idesc(T::kAbFormat, a_mn, b_mn, T::BM,
                     (T::kConv == Conv::kSplit3 || T::kConv == Conv::kSplit4 || T::kConv == Conv::kSplit3M)
                         ? 2 * T::BN
                         : T::BN);
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(p, t);
        const int ck = p.chunk_kb > 0 ? p.chunk_kb : (tc.kb1 - tc.kb0);
        for (int c0 = tc.kb0; c0 < tc.kb1 && ok; c0 += ck, ++g) {
          const int c1 = min(tc.kb1, c0 + ck);
          const uint32_t ab = g % T::kAccBufs;
          const uint32_t aph = (g / T::kAccBufs) & 1u;
          if (!mbar_wait(&acc_empty[ab], aph ^ 1u, ctl)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t d0 = tmem_base + ab * T::kAccStride;
          for (int kb = c0; kb < c1; ++kb, ++it) {
            const uint32_t st = it % T::kStagesOp;
            const uint32_t ph = (it / T::kStagesOp) & 1u;
            if (!mbar_wait(&op_full[st], ph, ctl)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t a_hi = op_smem + st * T::kOpStage;
            const uint32_t a_lo = a_hi + T::kATile;                       // split only
            const uint32_t b_hi = a_hi + T::kCopiesA * T::kATile;
            const uint32_t b_lo = b_hi + T::kBTile;                       // split only
#pragma unroll
            for (int ks = 0; ks < T::kKSteps; ++ks) {
              const uint32_t acc = (kb > c0 || ks > 0) ? 1u : 0u;
              const uint64_t da_hi = operand_desc<T>(a_hi, a_mn, ks);
              const uint64_t db_hi = operand_desc<T>(b_hi, b_mn, ks);
              if constexpr (T::kOp == Op::kTF32) {
                mma_tf32(d0, da_hi, db_hi, idesc_n, acc);
              } else if constexpr (T::kConv == Conv::kSplit3) {
                // [hh | hl] = A_hi * [B_hi | B_lo]  (B_hi and B_lo are adjacent)
                mma_f16(d0, da_hi, db_hi, idesc_2n, acc);
                // lh = A_lo * B_hi
                mma_f16(d0 + 2 * T::BN, operand_desc<T>(a_lo, a_mn, ks), db_hi, idesc_n, acc);
              } else if constexpr (T::kConv == Conv::kSplit3M) {
                // [hh | hl] = A_hi * [B_hi | B_lo];  then lh adds into hl's columns
                // (issued after the instruction that starts them, so always accumulating)
                mma_f16(d0, da_hi, db_hi, idesc_2n, acc);
                mma_f16(d0 + T::BN, operand_desc<T>(a_lo, a_mn, ks), db_hi, idesc_n, 1u);
              } else if constexpr (T::kConv == Conv::kSplit4) {
                // [hh | hl] = A_hi * [B_hi | B_lo];  [lh | ll] = A_lo * [B_hi | B_lo]
                mma_f16(d0, da_hi, db_hi, idesc_2n, acc);
                mma_f16(d0 + 2 * T::BN, operand_desc<T>(a_lo, a_mn, ks), db_hi, idesc_2n, acc);
              } else if constexpr (T::kConv == Conv::kSplitA2) {
                // two chains: A_hi B and A_lo B (B single)
                mma_f16(d0, da_hi, db_hi, idesc_n, acc);
                mma_f16(d0 + T::BN, operand_desc<T>(a_lo, a_mn, ks), db_hi, idesc_n, acc);
              } else if constexpr (T::kConv == Conv::kSplit1) {
                // one chain: hh, hl and lh all accumulate into the same columns
                mma_f16(d0, da_hi, db_hi, idesc_n, acc);
                mma_f16(d0, da_hi, operand_desc<T>(b_lo, b_mn, ks), idesc_n, 1u);
                mma_f16(d0, operand_desc<T>(a_lo, a_mn, ks), db_hi, idesc_n, 1u);
              } else {
                mma_f16(d0, da_hi, db_hi, idesc_n, acc);
              }
            }
            mma_commit(&op_empty[st]);
          }
          if (!ok) break;
          mma_commit(&acc_full[ab]);
        }
      }
      // wait for every MMA this thread issued before TMEM is released
      mma_commit(done_bar);
      drain_wait(done_bar, 0, p.wait_limit_ns);
    }
  } else if (warp < T::kConvWarp0) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    float* stg = epi_base + (warp - 2) * 1024;
    // warps sharing a lane quarter split the tile's 32-column chunks
    constexpr int kColGroups = T::kEpiWarps / 4;
    constexpr int kCcPer = T::BN / 32 / kColGroups;
    static_assert(kCcPer >= 1 && (T::BN / 32) % kColGroups == 0, "epilogue column split");
    const int cc0 = ((warp - 2) / 4) * kCcPer;
    const uint32_t stg_addr = smem_addr(stg);
    uint32_t g = 0;   // accumulation chunk, in the MMA warp's order
    bool ok = true;
    bool stores_pending = false;   // a TMA store may still be reading this warp's staging buffer
    for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
      const TileCoord tc = decode_tile(p, t);
      const int ck = p.chunk_kb > 0 ? p.chunk_kb : (tc.kb1 - tc.kb0);
      const int nchunks = (tc.kb1 - tc.kb0 + ck - 1) / ck;
      void* out;          // element (r, c) at out[r * ldo + c], type out_dt
      int64_t ldo;
      float alpha, beta;
      bool vec_ok;
      int out_dt;
      if (p.splits > 1) {
        out = p.partial + ((int64_t)tc.s * p.batch + tc.b) * (int64_t)p.m * p.n;
        ldo = p.n;
        alpha = 1.0f;
        beta = 0.0f;
        vec_ok = p.p_vec_ok != 0;
        out_dt = kOutF32;
      } else {
        out = static_cast<uint8_t*>(p.c) + (int64_t)tc.b * p.stride_c * (p.c_dtype == kOutF32 ? 4 : 2);
        ldo = p.ldc;
        alpha = p.alpha;
        beta = p.beta;
        vec_ok = p.c_vec_ok != 0;
        out_dt = p.c_dtype;
      }
      const int row_base = tc.mb * T::BM + 32 * q;
#pragma unroll 1
      for (int ci = 0; ci < nchunks; ++ci, ++g) {
        const uint32_t ab = g % T::kAccBufs;
        const uint32_t aph = (g / T::kAccBufs) & 1u;
        if (!warp_wait(&acc_full[ab], aph, ctl)) { ok = false; break; }
        tc_fence_after_sync();
        const uint32_t tacc = tmem_base + lane_off + ab * T::kAccStride;
        const uint32_t trun = tmem_base + lane_off + T::kRunBase;
        const bool last = (ci == nchunks - 1);
        const bool have_run = (ci > 0);
  #pragma unroll 1
        for (int cc = cc0; cc < cc0 + kCcPer; ++cc) {
          float v[32];
          if constexpr (T::kPromote) {
            // chunk total of the split's chains, plus the running sum of the
            // earlier chunks of this tile
  #pragma unroll
            for (int h = 0; h < 2; ++h) {
              float x0[16], x1[16], x2[16], x3[16], r[16];
              const uint32_t col = cc * 32 + h * 16;
              tmem_ld_16cols(tacc + col, x0);
              tmem_ld_16cols(tacc + T::BN + col, x1);
              if constexpr (T::kConv == Conv::kSplit3 || T::kConv == Conv::kSplit4)
                tmem_ld_16cols(tacc + 2 * T::BN + col, x2);
              if constexpr (T::kConv == Conv::kSplit4) tmem_ld_16cols(tacc + 3 * T::BN + col, x3);
              if (have_run) tmem_ld_16cols(trun + col, r);
              tmem_ld_wait();
              if (h == 1 && cc == cc0 + kCcPer - 1) {
                // this warp's share of the chains is in registers: the next
                // chunk's MMAs may overwrite them while the running sum (in
                // columns of its own) is updated
                tc_fence_before_sync();
                mbar_arrive(&acc_empty[ab]);
              }
              // 2^-L undoes the lo half's scale (exact: a power of two)
              const float lo_inv = p.lo_inv;
  #pragma unroll
              for (int j = 0; j < 16; ++j) {
                // three chains: hh + 2^-L (hl + lh); two chains (A-only split): hb + 2^-L lb
                float x;
                if constexpr (T::kConv == Conv::kSplit4)   // ... + 2^-2L ll
                  x = x0[j] + (lo_inv * (x1[j] + x2[j]) + (lo_inv * lo_inv) * x3[j]);
                else if constexpr (T::kConv == Conv::kSplit3)
                  x = x0[j] + lo_inv * (x1[j] + x2[j]);
                else
                  x = x0[j] + lo_inv * x1[j];
                v[h * 16 + j] = have_run ? r[j] + x : x;
              }
            }
            if (!last) {
              tmem_st_16cols(trun + cc * 32, v);
              tmem_st_16cols(trun + cc * 32 + 16, v + 16);
              // the next fold reads these columns back
              if (cc == cc0 + kCcPer - 1) tmem_st_wait();
            }
          } else if constexpr (T::kConv == Conv::kSplit3M) {
            // hh + 2^-L (hl + lh), the lo products' sum from their shared accumulator
            const float lo_inv = p.lo_inv;
  #pragma unroll
            for (int h = 0; h < 2; ++h) {
              float x0[16], x1[16];
              const uint32_t col = cc * 32 + h * 16;
              tmem_ld_16cols(tacc + col, x0);
              tmem_ld_16cols(tacc + T::BN + col, x1);
              tmem_ld_wait();
              if (h == 1 && cc == cc0 + kCcPer - 1) {
                tc_fence_before_sync();
                mbar_arrive(&acc_empty[ab]);
              }
  #pragma unroll
              for (int j = 0; j < 16; ++j) v[h * 16 + j] = x0[j] + lo_inv * x1[j];
            }
          } else {
            tmem_ld_32cols(tacc + cc * 32, v);
            tmem_ld_wait();
            if (cc == cc0 + kCcPer - 1) {
              // this warp's share of the accumulator is in registers
              tc_fence_before_sync();
              mbar_arrive(&acc_empty[ab]);
            }
          }
          if (!last) continue;   // chunk folded into the running sum; nothing to store yet
          const int col_base = tc.nb * T::BN + cc * 32;
          if (row_base >= p.m || col_base >= p.n) continue;
          if (p.tma_store) {
            // The staging image is the 128-byte swizzle of a 32 x 32 fp32 box:
            // one TMA store writes the block (rows past m and columns past n
            // are not written).  alpha * acc, as the register path stores it.
            if (stores_pending) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
  #pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= alpha;
            stage_write_row(stg_addr, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int z = p.splits > 1 ? tc.s * p.batch + tc.b : tc.b;
              tma_store_3d(&p.map_out, stg_addr, col_base, row_base, z);
              bulk_commit();
            }
            stores_pending = true;
            continue;
          }
          // transpose through a per-warp swizzled 32x32 staging tile so that
          // global stores are row-contiguous
          stage_write_row(stg_addr, lane, v);
          __syncwarp();
          if (vec_ok && col_base + 32 <= p.n) {
  #pragma unroll
            for (int it = 0; it < 8; ++it) {
              const int r = it * 4 + (lane >> 3);
              const int ch = lane & 7;
              const float4 x = stage_read_chunk(stg_addr, lane, it);
              const int grow = row_base + r;
              if (grow < p.m) {
                const int64_t idx = (int64_t)grow * ldo + col_base + ch * 4;
                float4 o;
                if (beta != 0.0f) {
                  const float4 c0 = out_load4(out, idx, out_dt);
                  o.x = fmaf(beta, c0.x, alpha * x.x);
                  o.y = fmaf(beta, c0.y, alpha * x.y);
                  o.z = fmaf(beta, c0.z, alpha * x.z);
                  o.w = fmaf(beta, c0.w, alpha * x.w);
                } else {
                  o.x = alpha * x.x;
                  o.y = alpha * x.y;
                  o.z = alpha * x.z;
                  o.w = alpha * x.w;
                }
                out_store4(out, idx, o, out_dt);
              }
            }
          } else {
            const int gcol = col_base + lane;
  #pragma unroll 4
            for (int r = 0; r < 32; ++r) {
              const float x = stage_read_elem(stg_addr, lane, r);
              const int grow = row_base + r;
              if (grow < p.m && gcol < p.n) {
                const int64_t idx = (int64_t)grow * ldo + gcol;
                out_store(out, idx, (beta != 0.0f) ? fmaf(beta, out_load(out, idx, out_dt), alpha * x) : alpha * x,
                          out_dt);
              }
            }
          }
          __syncwarp();
        }
      }
    }
    // this warp's TMA stores complete before the CTA may exit
    if (stores_pending && lane == 0) bulk_wait_all();
    __syncwarp();
  } else {
    // ------------------------------------------------------------ converters
    if constexpr (T::kHasConv) {
      const int ct = threadIdx.x - T::kConvWarp0 * 32;
      constexpr int kChunks = (T::BM + T::BN) * 8;  // 4-element chunks per stage
      constexpr int kPerThread = kChunks / T::kConvThreads;
      static_assert(kChunks % T::kConvThreads == 0, "chunk split");
      using SE = SrcElem<T::kSrcT>;
      using E = typename SE::type;
      const E* __restrict__ ga = reinterpret_cast<const E*>(p.a);
      const E* __restrict__ gb = reinterpret_cast<const E*>(p.b);
      // Raw source values of one stage for this thread: fp32 values, or
      // 16-bit codes (4 per chunk).
      struct Raw {
        float x[kPerThread][4];
        unsigned short h[kPerThread][4];
      };
      // Generic source: read this thread's chunks of stage (tc, kb) from
      // global memory (zero outside the matrix).
      auto gather = [&](const TileCoord& tc, int kb, Raw& raw) {
        const int k0 = kb * T::BK;
#pragma unroll
        for (int i = 0; i < kPerThread; ++i) {
          const int wi = ct + i * T::kConvThreads;
          const bool isA = wi < T::BM * 8;
          const int wl = isA ? wi : wi - T::BM * 8;
          const uint32_t lg = wl >> 3, ch = wl & 7;
          const bool mn = isA ? p.a_mn_major : p.b_mn_major;
          const int rows_lim = isA ? p.m : p.n;
          const int row0 = isA ? tc.mb * T::BM : tc.nb * T::BN;
          const int64_t ld = isA ? p.lda : p.ldb;
          const E* g = (isA ? ga : gb) + (int64_t)tc.b * (isA ? p.stride_a : p.stride_b);
          // the chunk's 4 elements are consecutive in memory: (row r0,
          // k kk0..kk0+3) for K-major, (rows r0..r0+3, k kk0) for MN-major
          int r0, kk0;
          if (!mn) {
            r0 = row0 + (int)lg;
            kk0 = k0 + (int)ch * 4;
          } else {
            r0 = row0 + (int)(lg / T::BK) * T::BK + (int)ch * 4;
            kk0 = k0 + (int)(lg % T::BK);
          }
          const int64_t idx0 = mn ? (int64_t)kk0 * ld + r0 : (int64_t)r0 * ld + kk0;
          const bool whole = mn ? (r0 + 3 < rows_lim && kk0 < p.k) : (r0 < rows_lim && kk0 + 3 < p.k);
          if (whole && (isA ? p.a_vec_ok : p.b_vec_ok)) {
            // one aligned vector load (16 bytes of fp32, 8 of 16-bit codes)
            if constexpr (T::kSrcT == SrcT::kF32) {
              const float4 v = __ldg(reinterpret_cast<const float4*>(g + idx0));
              raw.x[i][0] = v.x; raw.x[i][1] = v.y; raw.x[i][2] = v.z; raw.x[i][3] = v.w;
              raw.h[i][0] = raw.h[i][1] = raw.h[i][2] = raw.h[i][3] = 0;
            } else {
              const uint2 v = __ldg(reinterpret_cast<const uint2*>(g + idx0));
              raw.h[i][0] = (unsigned short)(v.x & 0xFFFFu); raw.h[i][1] = (unsigned short)(v.x >> 16);
              raw.h[i][2] = (unsigned short)(v.y & 0xFFFFu); raw.h[i][3] = (unsigned short)(v.y >> 16);
              raw.x[i][0] = raw.x[i][1] = raw.x[i][2] = raw.x[i][3] = 0.0f;
            }
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int r = mn ? r0 + e : r0;
              const int kk = mn ? kk0 : kk0 + e;
              const bool in = (r < rows_lim) && (kk < p.k);
              const int64_t idx = idx0 + e;
              if constexpr (T::kSrcT == SrcT::kF32) {
                raw.x[i][e] = in ? SE::load(g + idx) : 0.0f;
                raw.h[i][e] = 0;
              } else {
                raw.h[i][e] = in ? SE::load(g + idx) : (unsigned short)0;
                raw.x[i][e] = 0.0f;
              }
            }
          }
        }
      };
      // The generic source issues the next stage's loads before converting
      // and storing the current one, so that one stage's global-memory
      // latency overlaps the work of the previous stage.
      Raw cur, nxt;
      if constexpr (T::kSrc == Src::kGeneric) {
        if ((int)blockIdx.x < p.num_tiles) {
          const TileCoord tc = decode_tile(p, blockIdx.x);
          if (tc.kb0 < tc.kb1) gather(tc, tc.kb0, cur);
        }
      }
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(p, t);
        for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++it) {
          // the staging ring (read) and the operand ring (written) turn at
          // their own depths
          const uint32_t ss = T::kStaged ? it % T::kStagesStg : 0u;
          const uint32_t sph = T::kStaged ? (it / T::kStagesStg) & 1u : 0u;
          const uint32_t st = it % T::kStagesOp;
          const uint32_t ph = (it / T::kStagesOp) & 1u;
          if constexpr (T::kSrc == Src::kGeneric) {
            if (kb + 1 < tc.kb1) {
              gather(tc, kb + 1, nxt);
            } else {
              const int tn = t + (int)gridDim.x;
              if (tn < p.num_tiles) {
                const TileCoord tcn = decode_tile(p, tn);
                if (tcn.kb0 < tcn.kb1) gather(tcn, tcn.kb0, nxt);
              }
            }
          }
          if constexpr (T::kStaged) {
            if (!warp_wait(&stg_full[ss], sph, ctl)) { ok = false; break; }
          }
          uint32_t w[kPerThread][4];
          // ---- convert (staging written by TMA, 128B-swizzled fp32; or the
          //      values gathered from global memory) into packed operand words
#pragma unroll
          for (int i = 0; i < kPerThread; ++i) {
            const int wi = ct + i * T::kConvThreads;
            const bool isA = wi < T::BM * 8;
            const int wl = isA ? wi : wi - T::BM * 8;
            const uint32_t lg = wl >> 3, ch = wl & 7;
            float x[4];
            unsigned short h[4];
            if constexpr (T::kStaged) {
              const uint32_t base = stg_smem + ss * T::kStgStage + (isA ? 0u : (uint32_t)T::kStgATile);
              const float4 v = ld_shared_f4(base + swz_chunk_offset<128>(lg, ch));
              x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
              h[0] = h[1] = h[2] = h[3] = 0;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                x[e] = cur.x[i][e];
                h[e] = cur.h[i][e];
              }
            }
            pack_chunk<T>(x, h, isA ? p.scale_a : p.scale_b, p.lo_mul, w[i], isA);
          }
          if constexpr (T::kSrc == Src::kGeneric) cur = nxt;
          if constexpr (T::kStaged) {
            // The staging reads must have completed before the producer's
            // TMA (async proxy) refills this buffer: the conversion that
            // consumes them is register arithmetic the compiler may place
            // after the arrive, so nothing else orders the loads before it.
            // The proxy fence does; then hand the buffer back.
            fence_proxy_async_smem();
            mbar_arrive(&stg_empty[ss]);
          }
          if (!warp_wait(&op_empty[st], ph ^ 1u, ctl)) { ok = false; break; }
          // ---- scatter into the swizzled operand tiles
          const uint32_t a_hi = op_smem + st * T::kOpStage;
          const uint32_t b_hi = a_hi + T::kCopiesA * T::kATile;
#pragma unroll
          for (int i = 0; i < kPerThread; ++i) {
            const int wi = ct + i * T::kConvThreads;
            const bool isA = wi < T::BM * 8;
            const int wl = isA ? wi : wi - T::BM * 8;
            const uint32_t lg = wl >> 3, ch = wl & 7;
            const uint32_t hi_tile = isA ? a_hi : b_hi;
            const uint32_t lo_tile = hi_tile + (isA ? (uint32_t)T::kATile : (uint32_t)T::kBTile);
            store_chunk<T>(w[i], hi_tile, lo_tile, lg, ch, isA ? (p.a_mn_major != 0) : (p.b_mn_major != 0), isA);
          }
          fence_proxy_async_smem();
          mbar_arrive(&op_full[st]);
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, T::kTmemCols);
  }
}

template <class T>
bool tc_fill(TcKernel* out) {
  out->fn = reinterpret_cast<const void*>(&tc_gemm_kernel<T>);
  out->block = T::kThreads;
  out->smem_bytes = T::kSmemBytes;
  out->bn = T::BN;
  return true;
}

}  // namespace mpg
