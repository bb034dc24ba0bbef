// Fused prompt attention on the tensor cores (sm_103a):
//     O = softmax(scale * Q K^T) V
// with the scores and the probabilities kept on chip ("qsa_prompt_attn:
// Volta m8n8k4 kernel - keep the hi and lo halves in separate accumulator
// chains", sections "What's going on" and "The fix").  q is split into an
// FP16 hi half and a lo half for q.k, p for p.v; K and V are FP16 (the
// key/value cache's storage type).  The hi and lo products accumulate in
// separate TMEM chains that are added in plain fp32 (the two-chain form), or
// in one chain (the single-chain form the fix replaced).
//
// One CTA takes 128 queries and a range of keys, in blocks of 96 keys:
//   warp 0      TMA producer: K and V blocks (96 keys x 128 dims, fp16,
//               128-byte swizzle) into separate rings of 2 stages (K released
//               once S_j has read it, V after O_j), K one block ahead of V
//   warp 1      TMEM allocation; lane 0 issues every MMA:
//                 S_j = [Q_hi ; Q_lo] K_j^T   (M 128, N 96, K 128) -> 2 chains
//                 O_j = [P_hi ; P_lo] V_j     (M 128, N 128, K 96) -> 2 chains
//               in the order S_(j+1), O_j: S has one TMEM buffer, and S_(j+1)
//               goes in as soon as the compute warps have read S_j, while
//               O_(j-1) still runs.  P's first 64 keys sit in a 128-byte
//               swizzled atom column, the last 32 in a 64-byte swizzled one.
//   warps 2-17  softmax and folds of O, four warps per TMEM lane quarter
//               (32 query rows); each of the four takes a quarter of a row:
//               24 of the block's keys for the softmax and 32 of the output
//               dims for the folds.
//               softmax of block j: s = (S_hi + 2^-11 S_lo) * scale * log2(e);
//               the four parts exchange their maxima (shared memory and an
//               mbarrier per lane quarter that all four parts arrive on,
//               waited on with the same bounded wait as every other handoff),
//               so all compute the same reference maximum m_ref.  m_ref
//               moves only when a block's maximum exceeds it by more than 8
//               (lazy rescaling: p = 2^(s - m_ref) <= 2^8, well inside
//               fp16); p is split into hi/lo fp16 and written to shared
//               memory as the A operand of the next MMA; each part keeps its
//               own running sum.
//               The O chains in TMEM accumulate the products of successive
//               blocks (all relative to m_ref).  A fold adds them to the fp32
//               running output in registers, O_run = O_run * 2^(r - m_ref) +
//               (O_hi + 2^-11 O_lo) * 2^(m_old - m_ref) (round to nearest),
//               and zeroes them; a warp folds after every fourth block, before
//               a block whose softmax moved m_ref in any of its rows, and at
//               the end.  A warp runs the softmax of block j+1 before the
//               fold of block j, so the tensor core always has the next
//               block's work.  At the end O = O_run / sum (or the
//               unnormalised partial with its m_ref and sum when the keys are
//               split across CTAs; a merge kernel combines the partials).
// First, the compute warps load the CTA's 128 x 128 fp32 block of Q and split it into
// the swizzled hi/lo operand tiles.  Every wait is bounded.
#include "tc_gemm.cuh"

namespace mpg {
namespace {

template <bool kTwoChain, int PARTS>
struct AttnTraits {
  static constexpr int BM = 128;     // queries per CTA
  static constexpr int BKEY = kAttnKeyBlock;   // keys per block (96)
  static_assert(BKEY == 96, "the P tile's two swizzle regions and the 24-key parts assume 96");
  static constexpr int D = 128;      // head dimension (q.k and v)
  static constexpr int kKStages = 2;
  static constexpr int kVStages = 2;
  static constexpr int kQTile = BM * D * 2;          // 32 KB per half (hi or lo)
  static constexpr int kKVTile = BKEY * D * 2;       // 24 KB (K or V block): two 64-dim halves
  // P, the A operand of O = P V (K-major, keys contiguous): keys 0-63 in a
  // 128-byte swizzled atom column (16 KB), keys 64-95 in a 64-byte swizzled
  // one (8 KB)
  static constexpr int kPCol0 = BM * 128;
  static constexpr int kPTile = BM * 128 + BM * 64;  // 24 KB per half
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + 2 * kQTile;
  static constexpr int kOffV = kOffK + kKStages * kKVTile;
  static constexpr int kOffP = kOffV + kVStages * kKVTile;
  // compute warps: PARTS warps share each TMEM lane quarter (32 query rows);
  // each takes KP of a block's keys and DP of the output dims of its rows
  static constexpr int kParts = PARTS;
  static constexpr int kComputeThreads = 4 * PARTS * 32;
  static constexpr int KP = BKEY / PARTS;
  static constexpr int DP = D / PARTS;
  static constexpr int kOffMax = kOffP + 2 * kPTile;            // [block parity][part][128] partial maxima
  static constexpr int kOffSum = kOffMax + 2 * PARTS * BM * 4;  // [part][128] partial sums
  static constexpr int kOffBars = kOffSum + PARTS * BM * 4;
  static constexpr int kNumBars = 2 * kKStages + 2 * kVStages + 1 + 1 + 2 + 2 + 1 + 1 + 4;
  static constexpr int kSmemBytes = 1024 + kOffBars + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr int kThreads = 64 + kComputeThreads;
  // TMEM columns
  static constexpr uint32_t kColS = 0;      // S: hi at 0, lo at BKEY
  static constexpr uint32_t kColOhi = 256;
  static constexpr uint32_t kColOlo = 384;
  static constexpr int kL = kTwoChain ? 11 : 0;   // lo scale exponent of the split
};

constexpr float kLoScale = 0x1p-11f;
// Lazy rescaling of the online softmax: the reference maximum moves only
// when a block's maximum exceeds it by more than kLazyLog2, so p <= 2^8.
constexpr float kLazyLog2 = 8.0f;
// Blocks of products the O chains accumulate in TMEM between folds into the
// fp32 running output (384 keys: the tensor cores' own accumulation stays
// short, like the split GEMM's K chunks).
constexpr int kFoldBlocks = 4;

// 2^x by the hardware's approximate base-2 exponential (ex2.approx, results
// below 2^-126 flushed to zero: such probabilities add nothing to a sum
// of terms of which the largest is 1).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// K-major operand tile of `rows` lines whose K extent spans 128-byte atom
// columns stored one after another (each rows x 128 bytes); k-step `ks` of
// 16 fp16 elements.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, uint32_t rows, int ks) {
  return make_smem_desc(base + (uint32_t)(ks >> 2) * rows * 128u + (uint32_t)(ks & 3) * 32u, 16u, 1024u,
                        kSwizzle128B);
}
// MN-major (N contiguous) B tile: regions of 64 N x `lines` k-lines, one
// after the other.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, uint32_t lines, int ks) {
  return make_smem_desc(base + (uint32_t)ks * 16u * 128u, lines * 128u, 1024u, kSwizzle128B);
}
// K-major A tile of 128 rows whose first 64 k sit in a 128-byte swizzled
// atom column and the rest in a 64-byte swizzled one (the P tile).
__device__ __forceinline__ uint64_t p_desc(uint32_t base, uint32_t col0_bytes, int ks) {
  if (ks < 4) return make_smem_desc(base + (uint32_t)ks * 32u, 16u, 1024u, kSwizzle128B);
  return make_smem_desc(base + col0_bytes + (uint32_t)(ks - 4) * 32u, 16u, 512u, kSwizzle64B);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1) {
  tma_load_3d(dst, map, bar, c0, c1, 0);
}

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* q_tiles = smem + T::kOffQ;      // [hi | lo], each [2 atom columns][128 rows][128 B]
  uint8_t* k_tiles = smem + T::kOffK;      // stage s of each ring: [2 dim halves][BKEY keys][128 B]
  uint8_t* v_tiles = smem + T::kOffV;
  uint8_t* p_tiles = smem + T::kOffP;      // [hi | lo], each [128 rows][128 B] + [128 rows][64 B]
  float* part_max = reinterpret_cast<float*>(smem + T::kOffMax);
  float* part_sum = reinterpret_cast<float*>(smem + T::kOffSum);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::kOffBars);
  uint64_t* k_full = bars;
  uint64_t* k_empty = k_full + T::kKStages;
  uint64_t* v_full = k_empty + T::kKStages;
  uint64_t* v_empty = v_full + T::kVStages;
  uint64_t* s_full = v_empty + T::kVStages;
  uint64_t* s_empty = s_full + 1;
  uint64_t* p_full = s_empty + 1;           // [0] p_full, [1] p_empty
  uint64_t* p_empty = p_full + 1;
  uint64_t* o_full = p_full + 2;            // [0] o_full, [1] o_empty
  uint64_t* o_empty = o_full + 1;
  uint64_t* q_ready = o_full + 2;
  uint64_t* done_bar = q_ready + 1;
  uint64_t* xchg = done_bar + 1;            // [4]: the parts of a lane quarter exchange values
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xchg + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qb = blockIdx.x % p.num_q_blk;      // query block
  const int split = blockIdx.x / p.num_q_blk;   // key range
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(kb0 + p.kb_per_split, (p.lk + T::BKEY - 1) / T::BKEY);
  const int nb = kb1 - kb0;                    // >= 1 (the host never launches an empty range)

  if (threadIdx.x == 0) {
    for (int i = 0; i < T::kKStages; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    for (int i = 0; i < T::kVStages; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, T::kComputeThreads);
    mbar_init(p_full, T::kComputeThreads);
    mbar_init(p_empty, 1);
    mbar_init(o_full, 1);
    mbar_init(o_empty, T::kComputeThreads);
    mbar_init(q_ready, T::kComputeThreads);
    mbar_init(done_bar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&xchg[i], 32 * T::kParts);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  WaitCtl ctl;
  ctl.abort = abort_flag;
  ctl.status = p.status;
  ctl.limit_ns = p.wait_limit_ns;

  const uint32_t q_smem = smem_addr(q_tiles);
  const uint32_t k_smem = smem_addr(k_tiles);
  const uint32_t v_smem = smem_addr(v_tiles);
  const uint32_t p_smem = smem_addr(p_tiles);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&p.map_k);
      tma_prefetch_map(&p.map_v);
      // one block of a ring: wait for the stage, then the two 64-dim halves
      auto load = [&](const CUtensorMap* map, uint8_t* tiles, uint64_t* full, uint64_t* empty, int stages,
                      int j) -> bool {
        const int st = j % stages;
        if (!mbar_wait(&empty[st], ((j / stages) & 1u) ^ 1u, ctl)) return false;
        const int key0 = (kb0 + j) * T::BKEY;
        uint8_t* dst = tiles + st * T::kKVTile;
        mbar_arrive_expect_tx(&full[st], T::kKVTile);
        tma_load_2d(dst, map, &full[st], 0, key0);
        tma_load_2d(dst + T::kKVTile / 2, map, &full[st], 64, key0);
        return true;
      };
      int nk = 0, nv = 0;   // blocks issued on each ring
      bool ok = load(&p.map_k, k_tiles, k_full, k_empty, T::kKStages, 0);
      if (ok) nk = 1;
      for (int j = 0; j < nb && ok; ++j) {
        if (j + 1 < nb) {
          ok = load(&p.map_k, k_tiles, k_full, k_empty, T::kKStages, j + 1);
          if (!ok) break;
          nk = j + 2;
        }
        ok = load(&p.map_v, v_tiles, v_full, v_empty, T::kVStages, j);
        if (ok) nv = j + 1;
      }
      // copies issued must land before the CTA may exit
      for (int i = nk > T::kKStages ? nk - T::kKStages : 0; i < nk; ++i)
        drain_wait(&k_full[i % T::kKStages], (i / T::kKStages) & 1u, p.wait_limit_ns);
      for (int i = nv > T::kVStages ? nv - T::kVStages : 0; i < nv; ++i)
        drain_wait(&v_full[i % T::kVStages], (i / T::kVStages) & 1u, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc(0u, false, false, 128, T::BKEY);
      const uint32_t idesc_o = make_idesc(0u, false, true, 128, 128);
      const uint32_t q_hi = q_smem, q_lo = q_smem + T::kQTile;
      const uint32_t p_hi = p_smem, p_lo = p_smem + T::kPTile;
      bool ok = mbar_wait(q_ready, 0, ctl);
      tc_fence_after_sync();
      // one S buffer: S_j is issued once the compute warps have read S_(j-1)
      auto issue_s = [&](int j) -> bool {
        const uint32_t st = j % T::kKStages;
        if (!mbar_wait(&k_full[st], (j / T::kKStages) & 1u, ctl)) return false;
        if (!mbar_wait(s_empty, (j & 1u) ^ 1u, ctl)) return false;
        tc_fence_after_sync();
        const uint32_t kt = k_smem + st * T::kKVTile;
        const uint32_t d_hi = tmem_base + T::kColS;
#pragma unroll
        for (int ks = 0; ks < T::D / 16; ++ks) {
          const uint64_t bk = kmajor_desc(kt, T::BKEY, ks);
          mma_f16(d_hi, kmajor_desc(q_hi, 128, ks), bk, idesc_s, ks > 0 ? 1u : 0u);
          if constexpr (T::kL == 11) {
            mma_f16(d_hi + T::BKEY, kmajor_desc(q_lo, 128, ks), bk, idesc_s, ks > 0 ? 1u : 0u);
          } else {
            mma_f16(d_hi, kmajor_desc(q_lo, 128, ks), bk, idesc_s, 1u);
          }
        }
        mma_commit(s_full);
        mma_commit(&k_empty[st]);
        return true;
      };
      auto issue_o = [&](int j) -> bool {
        const uint32_t st = j % T::kVStages;
        if (!mbar_wait(p_full, j & 1u, ctl)) return false;
        if (!mbar_wait(&v_full[st], (j / T::kVStages) & 1u, ctl)) return false;
        if (!mbar_wait(o_empty, (j & 1u) ^ 1u, ctl)) return false;
        tc_fence_after_sync();
        const uint32_t vt = v_smem + st * T::kKVTile;
        const uint32_t d_hi = tmem_base + T::kColOhi, d_lo = tmem_base + T::kColOlo;
#pragma unroll
        for (int ks = 0; ks < T::BKEY / 16; ++ks) {
          const uint64_t bv = mnmajor_desc(vt, T::BKEY, ks);
          // O accumulates across blocks: the compute warps fold it into
          // registers (and zero it) every few blocks
          const uint32_t acc = (j > 0 || ks > 0) ? 1u : 0u;
          mma_f16(d_hi, p_desc(p_hi, T::kPCol0, ks), bv, idesc_o, acc);
          if constexpr (T::kL == 11) {
            mma_f16(d_lo, p_desc(p_lo, T::kPCol0, ks), bv, idesc_o, acc);
          } else {
            mma_f16(d_hi, p_desc(p_lo, T::kPCol0, ks), bv, idesc_o, 1u);
          }
        }
        mma_commit(o_full);
        mma_commit(p_empty);
        mma_commit(&v_empty[st]);
        return true;
      };
      // S_(j+1) goes in as soon as the compute warps have read S_j (while
      // O_(j-1) runs), then O_j once P_j is written
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nb && ok; ++j) {
        if (j + 1 < nb) ok = issue_s(j + 1);
        if (ok) ok = issue_o(j);
      }
      mma_commit(done_bar);
      drain_wait(done_bar, 0, p.wait_limit_ns);
    }
  } else {
    // ------------------------------------------------------------ Q split (compute warps)
    {
      // 128 rows x 16 chunks of 8 dims; each thread takes CPT consecutive chunks of one row
      constexpr int CPT = 2048 / T::kComputeThreads;
      const int ct = threadIdx.x - 64;
      const int row = ct / (16 / CPT);
      const int c0 = (ct % (16 / CPT)) * CPT;
      const int64_t grow = (int64_t)qb * T::BM + row;
      const float* src = p.q + grow * p.ldq;
#pragma unroll 1
      for (int c = c0; c < c0 + CPT; ++c) {
        float x[8];
        if (grow < p.lq) {
          if (p.q_vec_ok) {
            const float4 a = __ldg(reinterpret_cast<const float4*>(src + 8 * c));
            const float4 b = __ldg(reinterpret_cast<const float4*>(src + 8 * c + 4));
            x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __ldg(src + 8 * c + e);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[e] = 0.0f;
        }
        uint32_t h[4], l[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) split_pair<T::kL>(x[2 * e], x[2 * e + 1], 1.0f, h[e], l[e]);
        // dims 8c..8c+7: atom column c / 8, 16-byte chunk c % 8 of row `row`
        const uint32_t hi_base = q_smem + (uint32_t)(c >> 3) * T::BM * 128u;
        const uint32_t off = swz_chunk_offset<128>((uint32_t)row, (uint32_t)(c & 7));
        st_shared_v4(hi_base + off, h[0], h[1], h[2], h[3]);
        st_shared_v4(hi_base + T::kQTile + off, l[0], l[1], l[2], l[3]);
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    constexpr int KP = T::KP, DP = T::DP, NP = T::kParts;
    const int q4 = warp & 3;                      // TMEM lane quarter of this warp
    const int part = (warp - 2) >> 2;             // keys KP*part.., dims DP*part.. of the rows
    const int r = 32 * q4 + lane;                 // query row within the block
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    float o[DP];
#pragma unroll
    for (int i = 0; i < DP; ++i) o[i] = 0.0f;
    // m_ref: the reference maximum of the probabilities (p = 2^(s - m_ref))
    // and of the O chains accumulating in TMEM; it moves only when a block's
    // maximum exceeds it by more than kLazyLog2 (p stays <= 2^kLazyLog2).
    // o (registers) holds the folded blocks relative to r_reg.
    float m_ref = -INFINITY, r_reg = -INFINITY, l_part = 0.0f;
    uint32_t nx = 0;   // exchanges with the other parts of the rows so far
    bool ok = true;
    // step t: softmax of block t (t < nb), then correction of block t-1 (t >= 1)
    for (int t = 0; t <= nb && ok; ++t) {
      bool rescale = false;        // softmax of block t moved m_ref
      float o_ref = m_ref;         // the reference of the O chains in TMEM
      if (t < nb) {
        // ---------------------------------------------------------- softmax of block t
        const int j = t;
        if (!warp_wait(s_full, j & 1u, ctl)) { ok = false; break; }
        tc_fence_after_sync();
        float s[KP];
        const uint32_t t_hi = tmem_base + lane_off + T::kColS + (uint32_t)(KP * part);
        {
#pragma unroll
          for (int c = 0; c < KP / 8; ++c) tmem_ld_8cols(t_hi + 8 * c, s + 8 * c);
          if constexpr (T::kL == 11) {
            float lo[KP];
#pragma unroll
            for (int c = 0; c < KP / 8; ++c) tmem_ld_8cols(t_hi + T::BKEY + 8 * c, lo + 8 * c);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < KP; ++i) s[i] = (s[i] + kLoScale * lo[i]) * p.scale_log2;
          } else {
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < KP; ++i) s[i] = s[i] * p.scale_log2;
          }
        }
        tc_fence_before_sync();
        mbar_arrive(s_empty);
        // keys past the end of the sequence score -inf (only the last block
        // of the sequence has any)
        const int valid = p.lk - (kb0 + j) * T::BKEY - KP * part;
        if (valid < KP) {
#pragma unroll
          for (int i = 0; i < KP; ++i)
            if (i >= valid) s[i] = -INFINITY;
        }
        // maximum over this part's keys: eight running maxima, then a tree
        float tr[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) tr[i] = s[i];
#pragma unroll
        for (int i = 8; i < KP; ++i) tr[i & 7] = fmaxf(tr[i & 7], s[i]);
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) tr[i] = fmaxf(tr[i], tr[i + w]);
        // the parts of the row agree on the block's maximum
        float* mx = part_max + ((j & 1) * NP) * T::BM;
        mx[part * T::BM + r] = tr[0];
        mbar_arrive(&xchg[q4]);
        if (!warp_wait(&xchg[q4], nx & 1u, ctl)) { ok = false; break; }
        ++nx;
        float m_blk = mx[r];
#pragma unroll
        for (int k = 1; k < NP; ++k) m_blk = fmaxf(m_blk, mx[k * T::BM + r]);
        if (m_blk > m_ref + kLazyLog2) {   // always on the first block
          rescale = true;
          m_ref = m_blk;
        }
        const float alpha_l = exp2_approx(o_ref - m_ref);   // 1 unless m_ref moved; 0 on the first block
#pragma unroll
        for (int i = 0; i < KP; ++i) s[i] = exp2_approx(s[i] - m_ref);
        // sum: eight running sums, then a tree
#pragma unroll
        for (int i = 0; i < 8; ++i) tr[i] = s[i];
#pragma unroll
        for (int i = 8; i < KP; ++i) tr[i & 7] += s[i];
#pragma unroll
        for (int w = 4; w >= 1; w >>= 1)
#pragma unroll
          for (int i = 0; i < w; ++i) tr[i] += tr[i + w];
        l_part = l_part * alpha_l + tr[0];
        // p split into hi/lo fp16: this part's 8-key chunks of row r of the A
        // tiles (chunks 0-7 in the 128-byte swizzled column, 8-11 in the
        // 64-byte swizzled one)
        if (!warp_wait(p_empty, (j & 1u) ^ 1u, ctl)) { ok = false; break; }
        const uint32_t p_hi = p_smem, p_lo = p_smem + T::kPTile;
#pragma unroll
        for (int cc = 0; cc < KP / 8; ++cc) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            split_pair<T::kL>(s[8 * cc + 2 * e], s[8 * cc + 2 * e + 1], 1.0f, h[e], l[e]);
          const uint32_t c = (uint32_t)((KP / 8) * part + cc);
          const uint32_t off = c < 8 ? swz_chunk_offset<128>((uint32_t)r, c)
                                     : (uint32_t)T::kPCol0 + swz_chunk_offset<64>((uint32_t)r, c - 8);
          st_shared_v4(p_hi + off, h[0], h[1], h[2], h[3]);
          st_shared_v4(p_lo + off, l[0], l[1], l[2], l[3]);
        }
        fence_proxy_async_smem();
        mbar_arrive(p_full);
      }
      if (t >= 1) {
        // ---------------------------------------------------------- fold after block t-1
        // The O chains hold the blocks since the last fold, relative to
        // o_ref.  They are added to the registers (round to nearest, the
        // hi and lo chains summed in fp32) and zeroed every kFoldBlocks
        // blocks (bounding how long the tensor cores accumulate), before
        // block t's products when m_ref moved, and at the end; otherwise
        // the next block's products accumulate on top of them.
        const int j = t - 1;
        if (!warp_wait(o_full, j & 1u, ctl)) { ok = false; break; }
        // tcgen05.ld/st are warp-collective: the warp folds all its rows when
        // any of them moved its reference (for the others a_tm is 1)
        const bool fold = __any_sync(0xffffffffu, rescale) || t % kFoldBlocks == 0 || t == nb;
        if (fold) {
          tc_fence_after_sync();
          const uint32_t t_hi = tmem_base + lane_off + T::kColOhi + (uint32_t)(DP * part);
          const uint32_t t_lo = tmem_base + lane_off + T::kColOlo + (uint32_t)(DP * part);
          const float a_reg = exp2_approx(r_reg - m_ref);   // 0 before the first fold
          const float a_tm = exp2_approx(o_ref - m_ref);
          constexpr int CW = DP / 2;   // columns per TMEM load
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float a[CW];
            if constexpr (CW == 32) tmem_ld_32cols(t_hi + CW * c, a); else tmem_ld_16cols(t_hi + CW * c, a);
            if constexpr (T::kL == 11) {
              float e[CW];
              if constexpr (CW == 32) tmem_ld_32cols(t_lo + CW * c, e); else tmem_ld_16cols(t_lo + CW * c, e);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < CW; ++i) o[CW * c + i] = fmaf(o[CW * c + i], a_reg, (a[i] + kLoScale * e[i]) * a_tm);
            } else {
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < CW; ++i) o[CW * c + i] = fmaf(o[CW * c + i], a_reg, a[i] * a_tm);
            }
          }
          r_reg = m_ref;
          if (t < nb) {
            // the next block's products start the chains again
            float z[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) z[i] = 0.0f;
#pragma unroll
            for (int c = 0; c < DP / 16; ++c) {
              tmem_st_16cols(t_hi + 16 * c, z);
              if constexpr (T::kL == 11) tmem_st_16cols(t_lo + 16 * c, z);
            }
            tmem_st_wait();
          }
        }
        tc_fence_before_sync();
        mbar_arrive(o_empty);
      }
    }
    // the row's sum is the sum of its parts' sums
    if (ok) {
      part_sum[part * T::BM + r] = l_part;
      mbar_arrive(&xchg[q4]);
      ok = warp_wait(&xchg[q4], nx & 1u, ctl);
    }
    float l_row = 0.0f;
    if (ok) {
#pragma unroll
      for (int k = 0; k < NP; ++k) l_row += part_sum[k * T::BM + r];
    }
    const int64_t grow = (int64_t)qb * T::BM + r;
    if (ok && grow < p.lq) {
      if (p.splits == 1) {
        const float inv = 1.0f / l_row;
        float* dst = p.o + grow * p.ldo + DP * part;
#pragma unroll
        for (int i = 0; i < DP; ++i) dst[i] = o[i] * inv;
      } else {
        float* dst = p.part_o + ((int64_t)split * p.lq + grow) * 128 + DP * part;
#pragma unroll
        for (int i = 0; i < DP; i += 4) *reinterpret_cast<float4*>(dst + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        if (part == 0) {
          p.part_m[(int64_t)split * p.lq + grow] = m_ref;
          p.part_l[(int64_t)split * p.lq + grow] = l_row;
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, 512);
  }
}

// O[i, t] = sum_s Opart_s[i, t] 2^(m_s - M) / sum_s l_s 2^(m_s - M), M = max_s m_s
__global__ void attn_merge_kernel(const AttnParams p) {
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;   // (row, 4-dim group)
  if (idx >= (int64_t)p.lq * 32) return;
  const int64_t row = idx >> 5;
  const int t = (int)(idx & 31) * 4;
  float mx = -INFINITY;
  for (int s = 0; s < p.splits; ++s) mx = fmaxf(mx, p.part_m[(int64_t)s * p.lq + row]);
  float l = 0.0f;
  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  for (int s = 0; s < p.splits; ++s) {
    const float w = exp2f(p.part_m[(int64_t)s * p.lq + row] - mx);
    l = fmaf(p.part_l[(int64_t)s * p.lq + row], w, l);
    const float4 v = *reinterpret_cast<const float4*>(p.part_o + ((int64_t)s * p.lq + row) * 128 + t);
    acc.x = fmaf(v.x, w, acc.x);
    acc.y = fmaf(v.y, w, acc.y);
    acc.z = fmaf(v.z, w, acc.z);
    acc.w = fmaf(v.w, w, acc.w);
  }
  const float inv = 1.0f / l;
  float* dst = p.o + row * p.ldo + t;
  dst[0] = acc.x * inv;
  dst[1] = acc.y * inv;
  dst[2] = acc.z * inv;
  dst[3] = acc.w * inv;
}

template <class T>
cudaError_t launch_kernel(const AttnParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, T::kSmemBytes);
  if (e != cudaSuccess) return e;
  attn_kernel<T><<<p.num_q_blk * p.splits, T::kThreads, T::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

// warps per TMEM lane quarter of the compute warpgroups
constexpr int kAttnParts = 4;

int attention_smem_bytes() { return AttnTraits<true, kAttnParts>::kSmemBytes; }

cudaError_t launch_attention(const AttnParams& p, bool two_chain, cudaStream_t stream) {
  cudaError_t e = two_chain ? launch_kernel<AttnTraits<true, kAttnParts>>(p, stream)
                            : launch_kernel<AttnTraits<false, kAttnParts>>(p, stream);
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t items = (int64_t)p.lq * 32;
  attn_merge_kernel<<<(unsigned)((items + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mpg
