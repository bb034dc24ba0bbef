// The 16-bit and tf32 tensor-core product on a pair of CTAs (sm_103a,
// cta_group::2).
//
// A cluster of two CTAs on two SMs computes one 256 x 256 tile of C with
// tcgen05.mma.cta_group::2 (M = 256, N = 256): CTA rank r holds rows
// 128r .. 128r+127 of the tile's A panel and columns 128r .. 128r+127 of its B
// panel in shared memory, the tensor cores of the pair read both halves, and
// each CTA's TMEM receives its own 128 rows x 256 columns of the accumulator.
// Per SM this halves the B bytes that travel from L2 into shared memory (and
// that the tensor core reads back) for the same flops, compared with a
// 128 x 256 tile on one SM.  This is the GB300 counterpart of keeping the
// accumulator in registers and feeding it from swizzled shared memory
// ("tile_matmul(): use the cuBLASDx register-accumulator API ...", "Proposed
// change"): the operands are staged once per pair instead of once per SM.
//
// Roles (320 threads per CTA):
//   warp 0      TMA producer of this CTA's halves.  Both CTAs' copies signal
//               the rank-0 CTA's "full" barrier (cp.async.bulk.tensor
//               .cta_group::2), which expects the bytes of both.
//   warp 1      TMEM allocation (collective over the pair); on rank 0 its
//               lane 0 issues every MMA of the pair and commits with
//               multicast to both CTAs' barriers.
//   warps 2-9   epilogue of this CTA's 128 rows (two warps per TMEM lane
//               quarter, each taking half of the columns); they hand the
//               accumulator buffer back to rank 0 with a remote arrive.
//
// Every wait is bounded.  A timeout raises the abort flag of both CTAs, so
// the pair stops together; every role then drains what it has in flight and
// the pair meets at a final cluster barrier before TMEM is released.
#include <cstring>

#include "tc_gemm.cuh"

namespace mpg {
namespace {

template <Op O, Conv CV = Conv::kNone>
struct PairTraits {
  static constexpr Op kOp = O;
  // The three-chain split on the conversion pass's copies: the pair's tile
  // is 256 x 128.  One N = 256 instruction makes hh and hl at once: its B
  // operand [B_hi | B_lo] is split between the CTAs as the instruction
  // splits N, so CTA 0 holds B_hi (all 128 columns) and CTA 1 holds B_lo.
  // lh (N = 128) reads B_hi halved between the CTAs: each CTA also holds 64
  // of B_hi's columns.  Per SM and stage: A_hi, A_lo (128 rows each), one
  // whole B half and a quarter.
  static constexpr bool kSplit = (CV == Conv::kSplit3);
  static constexpr int BM = 128;    // rows of A held by one CTA
  static constexpr int BMP = 256;   // rows of the pair's tile
  static constexpr int BN = kSplit ? 128 : 256;    // columns of the pair's tile
  static constexpr int BNH = 128;   // B rows of one CTA's (first) B tile
  static constexpr int kOpBytes = (O == Op::kTF32) ? 4 : 2;
  static constexpr int BK = 128 / kOpBytes;   // one 128-byte line of k per stage (64, tf32 32)
  static constexpr int kRowBytes = 128;
  static constexpr uint32_t kSwizzle = kSwizzle128B;
  static constexpr int kInstrK = 32 / kOpBytes;   // k of one MMA: 16 (tf32 8)
  static constexpr int kKSteps = BK / kInstrK;
  static constexpr int kATile = BM * kRowBytes;
  static constexpr int kBTile = BNH * kRowBytes;
  static constexpr int kBHalfTile = (BN / 2) * kRowBytes;   // split: this CTA's half of B_hi for lh
  // plain: A half, B half (32 KB); split: A_hi, A_lo, B_hi or B_lo, B_hi half (56 KB)
  static constexpr int kOpStage = kSplit ? 2 * kATile + kBTile + kBHalfTile : kATile + kBTile;
  static constexpr int kStages = kSplit ? 3 : 6;
  static constexpr int kEpiWarps = 8;
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  // split: hh | hl (256 columns), lh (128), the running sum of the K chunks (128)
  static constexpr int kAccStride = kSplit ? 3 * BN : BN;
  static constexpr int kAccBufs = kSplit ? 1 : 2;
  static constexpr int kRunBase = kSplit ? 3 * BN : 0;
  static constexpr int kTmemCols = 512;
  static constexpr int kEpiBytes = kEpiWarps * 32 * 32 * 4;
  static constexpr int kNumBars = 2 * kStages + 2 * kAccBufs + 1;
  static constexpr int kSmemBytes = 1024 + kStages * kOpStage + kEpiBytes + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static_assert(kAccBufs * kAccStride + (kSplit ? BN : 0) <= kTmemCols, "TMEM budget");
  static_assert(!kSplit || O == Op::kF16, "the split's halves are fp16");
  static constexpr uint32_t kAbFormat = (O == Op::kF16) ? 0u : (O == Op::kBF16) ? 1u : 2u;
};

// ---------------------------------------------------------------------------
// cluster and cta_group::2 forms (used only by this kernel: every tcgen05
// instruction of one kernel has to name the same CTA group)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}

// Shared-window address of the same shared-memory location in CTA `rank` of
// the cluster.
__device__ __forceinline__ uint32_t cluster_smem_addr(uint32_t smem, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem), "r"(rank));
  return r;
}
// Generic address of the same location in CTA `rank` (distributed shared memory).
template <class T>
__device__ __forceinline__ T* cluster_generic_ptr(T* p, uint32_t rank) {
  uint64_t r;
  asm volatile("mapa.u64 %0, %1, %2;" : "=l"(r) : "l"(reinterpret_cast<uint64_t>(p)), "r"(rank));
  return reinterpret_cast<T*>(r);
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// 3-D tiled load into this CTA's shared memory; completion is signalled on
// the barrier at `bar_cluster_addr`, which may sit in the peer CTA.
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* map, uint32_t bar_cluster_addr,
                                                 int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster_addr), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

template <Op O>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  if constexpr (O == Op::kTF32) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// One arrival on the barrier at this offset in every CTA of `mask`, once all
// MMAs issued so far by this thread have completed.
__device__ __forceinline__ void mma_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_addr(bar)),
      "h"(mask)
      : "memory");
}

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1) tc_pair_kernel(const __grid_constant__ TcParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // Both CTAs run the same code on the same dynamic shared-memory layout, so
  // every buffer and barrier sits at the same offset in the two CTAs (the
  // MMA's descriptors and the multicast commits rely on it).
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* op_base = smem;
  float* epi_base = reinterpret_cast<float*>(op_base + T::kStages * T::kOpStage);
  uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(epi_base) + T::kEpiBytes);
  uint64_t* op_full = bars;                         // rank 0: both CTAs' halves of a stage landed
  uint64_t* op_empty = bars + T::kStages;           // each CTA: the pair's MMAs consumed the stage
  uint64_t* acc_full = bars + 2 * T::kStages;       // each CTA: accumulator buffer complete
  uint64_t* acc_empty = acc_full + T::kAccBufs;     // rank 0: both CTAs' epilogues drained it
  uint64_t* done_bar = acc_empty + T::kAccBufs;     // rank 0: every MMA of the pair finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t cid = cluster_id_x();
  const uint32_t ncl = num_clusters_x();

  if (threadIdx.x == 0) {
    for (int i = 0; i < T::kStages; ++i) {
      mbar_init(&op_full[i], 1);     // the rank-0 producer's arrive.expect_tx
      mbar_init(&op_empty[i], 1);    // one multicast commit
    }
    for (int i = 0; i < T::kAccBufs; ++i) {
      mbar_init(&acc_full[i], 1);                   // one multicast commit
      mbar_init(&acc_empty[i], 2 * T::kEpiWarps);   // one arrival per epilogue warp of the pair
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, T::kTmemCols);
    tmem_relinquish_pair();
    tc_fence_before_sync();
  }
  // barriers, abort flags and the TMEM address of both CTAs are in place
  // before either CTA touches the other's shared memory
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  // the set-up may overlap the end of the kernel that wrote the operands
  griddep_wait();
  griddep_launch_dependents();

  WaitCtl ctl;
  ctl.abort = abort_flag;
  ctl.peer_abort = cluster_generic_ptr(const_cast<int*>(abort_flag), rank ^ 1u);
  ctl.status = p.status;
  ctl.limit_ns = p.wait_limit_ns;

  const uint32_t op_smem = smem_addr(op_base);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&p.map_a);
      tma_prefetch_map(&p.map_b);
      const uint32_t full0 = cluster_smem_addr(smem_addr(op_full), 0);   // rank 0's op_full[0]
      constexpr int kRegion = T::BK * T::kRowBytes;                      // one MN-major region
      uint32_t it = 0;
      bool ok = true;
      for (int t = (int)cid; t < p.num_tiles && ok; t += (int)ncl) {
        const TileCoord tc = decode_item(p, t);
        for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++it) {
          const uint32_t st = it % T::kStages;
          const uint32_t ph = (it / T::kStages) & 1u;
          if (!mbar_wait(&op_empty[st], ph ^ 1u, ctl)) { ok = false; break; }
          if (rank == 0) mbar_arrive_expect_tx(&op_full[st], 2 * T::kOpStage);
          uint8_t* dst = op_base + st * T::kOpStage;
          const uint32_t bar = full0 + st * 8u;
          const int k0 = kb * T::BK;
          auto load_half = [&](const CUtensorMap* map, uint8_t* d, bool mn, int row0, int rows) {
            if (!mn) {
              tma_load_3d_pair(d, map, bar, k0, row0, tc.b);
            } else {
              for (int g = 0; g < rows / T::BK; ++g) tma_load_3d_pair(d + g * kRegion, map, bar, row0 + g * T::BK, k0, tc.b);
            }
          };
          if constexpr (T::kSplit) {
            // A_hi, A_lo (this CTA's rows); B_hi (rank 0) or B_lo (rank 1), all
            // of the tile's columns, in the 64-row boxes of the maps; this
            // CTA's half of B_hi's columns
            const int arow = tc.mb * T::BMP + (int)rank * T::BM;
            load_half(&p.map_a, dst, p.a_mn_major != 0, arow, T::BM);
            load_half(&p.map_a_lo, dst + T::kATile, p.a_mn_major != 0, arow, T::BM);
            const CUtensorMap* bx = rank == 0 ? &p.map_b : &p.map_b_lo;
            uint8_t* bdst = dst + 2 * T::kATile;
            if (p.b_mn_major) {
              load_half(bx, bdst, true, tc.nb * T::BN, T::BN);
            } else {
              for (int h = 0; h < 2; ++h)
                load_half(bx, bdst + h * T::kBHalfTile, false, tc.nb * T::BN + h * (T::BN / 2), T::BN / 2);
            }
            load_half(&p.map_b, bdst + T::kBTile, p.b_mn_major != 0, tc.nb * T::BN + (int)rank * (T::BN / 2),
                      T::BN / 2);
          } else {
            load_half(&p.map_a, dst, p.a_mn_major != 0, tc.mb * T::BMP + (int)rank * T::BM, T::BM);
            load_half(&p.map_b, dst + T::kATile, p.b_mn_major != 0, tc.nb * T::BN + (int)rank * T::BNH, T::BNH);
          }
        }
      }
      // A stage is released (op_empty) only after both halves landed and the
      // pair's MMAs read them, so waiting for the last releases also covers
      // this CTA's copies still in flight.
      const uint32_t n_drain = it < (uint32_t)T::kStages ? it : (uint32_t)T::kStages;
      for (uint32_t i = it - n_drain; i < it; ++i)
        drain_wait(&op_empty[i % T::kStages], (i / T::kStages) & 1u, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if constexpr (T::kSplit) {
      if (lane == 0 && rank == 0) {
        // The split: per k-step [hh | hl] += A_hi [B_hi | B_lo] (N = 256) and
        // lh += A_lo B_hi (N = 128), in K chunks of chunk_kb k-blocks, each
        // chunk on fresh chains that the epilogue folds into its running sum.
        const bool a_mn = p.a_mn_major != 0;
        const bool b_mn = p.b_mn_major != 0;
        const uint32_t idesc_2n = make_idesc(T::kAbFormat, a_mn, b_mn, T::BMP, 2 * T::BN);
        const uint32_t idesc_n = make_idesc(T::kAbFormat, a_mn, b_mn, T::BMP, T::BN);
        uint32_t it = 0, g = 0;
        bool ok = true;
        for (int t = (int)cid; t < p.num_tiles && ok; t += (int)ncl) {
          const TileCoord tc = decode_item(p, t);
          const int ck = p.chunk_kb > 0 ? p.chunk_kb : (tc.kb1 - tc.kb0);
          for (int c0 = tc.kb0; c0 < tc.kb1 && ok; c0 += ck, ++g) {
            const int c1 = min(tc.kb1, c0 + ck);
            if (!mbar_wait(&acc_empty[0], (g & 1u) ^ 1u, ctl)) { ok = false; break; }
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            tc_fence_after_sync();
            const uint32_t d0 = tmem_base;
            for (int kb = c0; kb < c1; ++kb, ++it) {
              const uint32_t st = it % T::kStages;
              const uint32_t ph = (it / T::kStages) & 1u;
              if (!mbar_wait(&op_full[st], ph, ctl)) { ok = false; break; }
              tc_fence_after_sync();
              const uint32_t a_hi = op_smem + st * T::kOpStage;
              const uint32_t a_lo = a_hi + T::kATile;
              const uint32_t bx = a_hi + 2 * T::kATile;
              const uint32_t bh = bx + T::kBTile;
#pragma unroll
              for (int ks = 0; ks < T::kKSteps; ++ks) {
                const uint32_t acc = (kb > c0 || ks > 0) ? 1u : 0u;
                mma_pair<T::kOp>(d0, operand_desc<T>(a_hi, a_mn, ks), operand_desc<T>(bx, b_mn, ks), idesc_2n, acc);
                mma_pair<T::kOp>(d0 + 2 * T::BN, operand_desc<T>(a_lo, a_mn, ks), operand_desc<T>(bh, b_mn, ks),
                                 idesc_n, acc);
              }
              mma_commit_multicast(&op_empty[st], 0x3);
            }
            if (!ok) break;
            mma_commit_multicast(&acc_full[0], 0x3);
          }
        }
        mma_commit_multicast(done_bar, 0x1);
        drain_wait(done_bar, 0, p.wait_limit_ns);
      }
    } else if (lane == 0 && rank == 0) {
      const bool a_mn = p.a_mn_major != 0;
      const bool b_mn = p.b_mn_major != 0;
      const uint32_t idesc = make_idesc(T::kAbFormat, a_mn, b_mn, T::BMP, T::BN);
      uint32_t it = 0, g = 0;
      bool ok = true;
      for (int t = (int)cid; t < p.num_tiles && ok; t += (int)ncl, ++g) {
        const TileCoord tc = decode_item(p, t);
        const uint32_t ab = g % T::kAccBufs;
        const uint32_t aph = (g / T::kAccBufs) & 1u;
        if (!mbar_wait(&acc_empty[ab], aph ^ 1u, ctl)) { ok = false; break; }
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        tc_fence_after_sync();
        const uint32_t d0 = tmem_base + ab * T::kAccStride;
        for (int kb = tc.kb0; kb < tc.kb1; ++kb, ++it) {
          const uint32_t st = it % T::kStages;
          const uint32_t ph = (it / T::kStages) & 1u;
          if (!mbar_wait(&op_full[st], ph, ctl)) { ok = false; break; }
          tc_fence_after_sync();
          const uint32_t a_tile = op_smem + st * T::kOpStage;
          const uint32_t b_tile = a_tile + T::kATile;
#pragma unroll
          for (int ks = 0; ks < T::kKSteps; ++ks)
            mma_pair<T::kOp>(d0, operand_desc<T>(a_tile, a_mn, ks), operand_desc<T>(b_tile, b_mn, ks), idesc,
                         (kb > tc.kb0 || ks > 0) ? 1u : 0u);
          mma_commit_multicast(&op_empty[st], 0x3);
        }
        if (!ok) break;
        mma_commit_multicast(&acc_full[ab], 0x3);
      }
      // every MMA of the pair completes before either CTA releases TMEM
      mma_commit_multicast(done_bar, 0x1);
      drain_wait(done_bar, 0, p.wait_limit_ns);
    }
  } else if constexpr (T::kSplit) {
    // ------------------------------------------------------------ epilogue of the split
    // Each K chunk: hh + 2^-L (hl + lh) added to the running sum (TMEM
    // columns of its own, round to nearest in fp32); after the last chunk,
    // alpha * sum + beta * C in C's type.
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    float* stg = epi_base + (warp - 2) * 1024;
    const uint32_t stg_addr = smem_addr(stg);
    constexpr int kColGroups = T::kEpiWarps / 4;
    constexpr int kCcPer = T::BN / 32 / kColGroups;
    const int cc0 = ((warp - 2) / 4) * kCcPer;
    const uint32_t acc_empty0 = cluster_smem_addr(smem_addr(acc_empty), 0);
    const uint32_t tacc = tmem_base + lane_off;
    const uint32_t trun = tmem_base + lane_off + T::kRunBase;
    const float lo_inv = p.lo_inv;
    uint32_t g = 0;
    bool ok = true;
    for (int t = (int)cid; t < p.num_tiles && ok; t += (int)ncl) {
      const TileCoord tc = decode_item(p, t);
      const int ck = p.chunk_kb > 0 ? p.chunk_kb : (tc.kb1 - tc.kb0);
      const int nchunks = (tc.kb1 - tc.kb0 + ck - 1) / ck;
      void* out;
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
      const int row_base = tc.mb * T::BMP + (int)rank * T::BM + 32 * q;
#pragma unroll 1
      for (int ci = 0; ci < nchunks; ++ci, ++g) {
        if (!warp_wait(&acc_full[0], g & 1u, ctl)) { ok = false; break; }
        tc_fence_after_sync();
        const bool last = (ci == nchunks - 1);
#pragma unroll 1
        for (int cc = cc0; cc < cc0 + kCcPer; ++cc) {
          float v[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float x0[16], x1[16], x2[16], r[16];
            const uint32_t col = cc * 32 + h * 16;
            tmem_ld_16cols(tacc + col, x0);
            tmem_ld_16cols(tacc + T::BN + col, x1);
            tmem_ld_16cols(tacc + 2 * T::BN + col, x2);
            if (ci > 0) tmem_ld_16cols(trun + col, r);
            tmem_ld_wait();
            if (h == 1 && cc == cc0 + kCcPer - 1) {
              // this warp's share of the chains is in registers: hand the
              // accumulator back to rank 0 (the running sum has columns of its own)
              tc_fence_before_sync();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(acc_empty0);
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float x = x0[j] + lo_inv * (x1[j] + x2[j]);
              v[h * 16 + j] = ci > 0 ? r[j] + x : x;
            }
          }
          if (!last) {
            tmem_st_16cols(trun + cc * 32, v);
            tmem_st_16cols(trun + cc * 32 + 16, v + 16);
            if (cc == cc0 + kCcPer - 1) tmem_st_wait();
            continue;
          }
          const int col_base = tc.nb * T::BN + cc * 32;
          if (row_base >= p.m || col_base >= p.n) continue;
          stage_write_row(stg_addr, lane, v);
          __syncwarp();
          if (vec_ok && col_base + 32 <= p.n) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = i * 4 + (lane >> 3);
              const int ch = lane & 7;
              const float4 x = stage_read_chunk(stg_addr, lane, i);
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
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    float* stg = epi_base + (warp - 2) * 1024;
    const uint32_t stg_addr = smem_addr(stg);
    constexpr int kColGroups = T::kEpiWarps / 4;
    constexpr int kCcPer = T::BN / 32 / kColGroups;
    const int cc0 = ((warp - 2) / 4) * kCcPer;
    const uint32_t acc_empty0 = cluster_smem_addr(smem_addr(acc_empty), 0);   // rank 0's acc_empty[0]
    uint32_t g = 0;
    bool ok = true;
    for (int t = (int)cid; t < p.num_tiles && ok; t += (int)ncl, ++g) {
      const TileCoord tc = decode_item(p, t);
      void* out;
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
      const uint32_t ab = g % T::kAccBufs;
      const uint32_t aph = (g / T::kAccBufs) & 1u;
      if (!warp_wait(&acc_full[ab], aph, ctl)) { ok = false; break; }
      tc_fence_after_sync();
      const uint32_t tacc = tmem_base + lane_off + ab * T::kAccStride;
      const int row_base = tc.mb * T::BMP + (int)rank * T::BM + 32 * q;
      // hand this warp's share of the accumulator buffer back to rank 0
      auto release = [&]() {
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(acc_empty0 + ab * 8u);
      };
      // one 32-column chunk of this warp's 32 rows: alpha * v + beta * C
      // stored in C's type, rows staged through shared memory so that each
      // store instruction writes whole lines
      auto store_chunk = [&](const float* v, int cc) {
        const int col_base = tc.nb * T::BN + cc * 32;
        if (row_base >= p.m || col_base >= p.n) return;
        stage_write_row(stg_addr, lane, v);
        __syncwarp();
        if (vec_ok && col_base + 32 <= p.n) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = i * 4 + (lane >> 3);
            const int ch = lane & 7;
            const float4 x = stage_read_chunk(stg_addr, lane, i);
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
      };
      if (tc.tail < 0) {
#pragma unroll 1
        for (int cc = cc0; cc < cc0 + kCcPer; ++cc) {
          float v[32];
          tmem_ld_32cols(tacc + cc * 32, v);
          tmem_ld_wait();
          // the last chunk of this warp's share is in registers
          if (cc == cc0 + kCcPer - 1) release();
          store_chunk(v, cc);
        }
        continue;
      }
      // Half of the k range of a tile of the split tail.  Each warp writes
      // its 32 x 128 piece of partial sums (chunk-major, one float4 per lane
      // per store: whole lines) and counts itself; the second of the two
      // halves to arrive adds the first's piece to its own and stores C.
      // Both orders give the same sum (fp32 addition commutes).
      const size_t piece = ((size_t)tc.tail * 2 + rank) * T::kEpiWarps + (size_t)(warp - 2);
      constexpr int kPieceF4 = kCcPer * 8 * 32;
      float4* own = reinterpret_cast<float4*>(p.tail_ws) + (piece * 2 + (size_t)tc.half) * kPieceF4;
      const float4* other = reinterpret_cast<const float4*>(p.tail_ws) + (piece * 2 + (size_t)(tc.half ^ 1)) * kPieceF4;
#pragma unroll 1
      for (int j = 0; j < kCcPer; ++j) {
        float v[32];
        tmem_ld_32cols(tacc + (cc0 + j) * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 8; ++i)
          own[(j * 8 + i) * 32 + lane] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
      __threadfence();
      __syncwarp();
      uint32_t prev = 0;
      if (lane == 0) prev = atomicAdd(p.tail_cnt + piece, 1u);
      prev = __shfl_sync(0xffffffffu, prev, 0);
      if (prev == 0) {
        release();   // the other half finishes this piece
        continue;
      }
      __threadfence();
#pragma unroll 1
      for (int j = 0; j < kCcPer; ++j) {
        float v[32];
        tmem_ld_32cols(tacc + (cc0 + j) * 32, v);
        tmem_ld_wait();
        if (j == kCcPer - 1) release();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 o = __ldcg(other + (j * 8 + i) * 32 + lane);
          v[4 * i] += o.x;
          v[4 * i + 1] += o.y;
          v[4 * i + 2] += o.z;
          v[4 * i + 3] += o.w;
        }
        store_chunk(v, cc0 + j);
      }
    }
  }

  // Neither CTA releases TMEM or exits while the other may still address its
  // shared memory (remote arrivals, multicast commits, copies signalling rank
  // 0) or while MMAs of the pair are in flight.
  __syncwarp();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, T::kTmemCols);
  }
}

template <class T>
void pair_fill(TcKernel* out) {
  out->fn = reinterpret_cast<const void*>(&tc_pair_kernel<T>);
  out->block = T::kThreads;
  out->smem_bytes = T::kSmemBytes;
  out->bn = T::BN;
}

// Hardware check of the M = 256 (cta_group::2) accumulator map: a cluster of
// two CTAs runs one k-block (K = 64, four K = 16 instructions of kind::f16)
// with the pair kernels' operand layout and descriptors -- CTA r holds rows
// 128r .. 128r+127 of A and columns (n/2) r .. (n/2) r + n/2 - 1 of B -- and
// every warp of both CTAs copies out its raw tcgen05.ld.32x32b.x32
// registers, unscattered.
constexpr int kPairProbeK = 64;
constexpr int kPairProbeSmem = 1024 + 128 * 128 + 128 * 128 + 64;

__global__ void __launch_bounds__(128, 1) probe_tmem_pair_kernel(const uint16_t* __restrict__ A,
                                                                  const uint16_t* __restrict__ B, int n,
                                                                  float* __restrict__ D, uint32_t* status,
                                                                  uint64_t limit_ns) {
  using T = PairTraits<Op::kF16>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tile = smem;                 // 128 lines of 128 bytes (this CTA's rows of A)
  uint8_t* b_tile = smem + 128 * 128;     // n / 2 lines of 128 bytes (this CTA's columns of B)
  uint64_t* bar = reinterpret_cast<uint64_t*>(b_tile + 128 * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int nh = n / 2;

  const uint32_t a_addr = smem_addr(a_tile), b_addr = smem_addr(b_tile);
  for (int i = threadIdx.x; i < (128 + nh) * 8; i += blockDim.x) {
    const bool isA = i < 128 * 8;
    const int w = isA ? i : i - 128 * 8;
    const int line = w >> 3, ch = w & 7;
    const uint16_t* src = isA ? A + (size_t)(128 * rank + line) * kPairProbeK : B + (size_t)(nh * rank + line) * kPairProbeK;
    const uint4 v = *reinterpret_cast<const uint4*>(src + ch * 8);
    st_shared_v4((isA ? a_addr : b_addr) + swz_chunk_offset<128>(line, ch), v.x, v.y, v.z, v.w);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  const uint32_t ncols = n <= 64 ? 64 : n <= 128 ? 128 : 256;
  if (warp == 0) {
    tmem_alloc_pair(tmem_slot, ncols);
    tmem_relinquish_pair();
    tc_fence_before_sync();
  }
  // both CTAs' operands, barriers and TMEM are in place before rank 0 issues
  cluster_sync_all();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  WaitCtl ctl;
  ctl.abort = abort_flag;
  ctl.peer_abort = cluster_generic_ptr(const_cast<int*>(abort_flag), rank ^ 1u);
  ctl.status = status;
  ctl.limit_ns = limit_ns;

  if (rank == 0 && threadIdx.x == 0) {
    const uint32_t idesc = make_idesc(0u /* f16 */, false, false, 256, (uint32_t)n);
#pragma unroll
    for (int ks = 0; ks < T::kKSteps; ++ks)
      mma_pair<Op::kF16>(tmem_base, operand_desc<T>(a_addr, false, ks), operand_desc<T>(b_addr, false, ks), idesc,
                         ks > 0 ? 1u : 0u);
    mma_commit_multicast(bar, 0x3);
  }
  __syncwarp();
  const bool ok = warp_wait(bar, 0, ctl);
  tc_fence_after_sync();
  if (ok) {
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    for (int c = 0; c < n / 32; ++c) {
      float v[32];
      tmem_ld_32cols(tmem_base + lane_off + c * 32, v);
      tmem_ld_wait();
      float* out = D + ((size_t)((rank * 4 + warp) * 32 + lane) * (n / 32) + c) * 32;
#pragma unroll
      for (int r = 0; r < 32; ++r) out[r] = v[r];
    }
  } else if (rank == 0) {
    drain_wait(bar, 0, limit_ns);   // the pair's MMAs may still run: let them finish
  }
  tc_fence_before_sync();
  __syncwarp();
  cluster_sync_all();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, ncols);
  }
}

}  // namespace

cudaError_t launch_probe_tmem_pair(const void* a, const void* b, int n, float* d, uint32_t* status,
                                   uint64_t limit_ns, cudaStream_t stream) {
  if (n != 64 && n != 128 && n != 256) return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(probe_tmem_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairProbeSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = kPairProbeSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const uint16_t* pa = static_cast<const uint16_t*>(a);
  const uint16_t* pb = static_cast<const uint16_t*>(b);
  e = cudaLaunchKernelEx(&cfg, probe_tmem_pair_kernel, pa, pb, n, d, status, limit_ns);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

bool tc_lookup_pair(Op op, Conv conv, TcKernel* out) {
  if (conv == Conv::kSplit3) {
    if (op != Op::kF16) return false;
    pair_fill<PairTraits<Op::kF16, Conv::kSplit3>>(out);
    return true;
  }
  if (conv != Conv::kNone) return false;
  switch (op) {
    case Op::kF16: pair_fill<PairTraits<Op::kF16>>(out); return true;
    case Op::kBF16: pair_fill<PairTraits<Op::kBF16>>(out); return true;
    case Op::kTF32: pair_fill<PairTraits<Op::kTF32>>(out); return true;
    default: return false;
  }
}

}  // namespace mpg
