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
// The scores are computed with the queries on the M side, the output
// transposed (head dimensions on M, queries on N):
//     S   = [Q_hi ; Q_lo] K^T     two chains of M 128 queries, N 128 keys, K 128 dims
//     O^T = V^T [P_hi ; P_lo]^T   M 128 dims, N 256 = 128 queries x (hi, lo), K 128 keys
// S keeps a query's scores in one TMEM lane, so the softmax's maxima and
// sums stay inside a thread; O^T puts the hi and lo chains of one k-step in a
// single N = 256 instruction (V^T is read once for both chains: 12 KB of
// shared memory per k-step instead of 16, the operand reads being what the
// tensor core waits on here), and P, written row by row, is its K-major B
// operand.  The single-chain form accumulates
// the hi and lo halves in one chain: S's lo products into the hi chain, O^T
// as two N = 128 instructions into one accumulator.
//
// One CTA takes 128 queries and a range of keys, in blocks of 128 keys:
//   warp 0      TMA producer: one ring of five 16 KB slots that K and V
//               share, filled in the order the MMAs read them: K_(j+1) (two
//               64-dim halves), then V_j (two 64-key halves).
//   warp 1      TMEM allocation; lane 0 issues every MMA, in the order S_(j+1),
//               O_j: S has one TMEM buffer (hi chain in columns 0-127, lo in
//               128-255), and S_(j+1) goes in as soon as the compute warps have
//               read S_j; O^T (columns 256-511) accumulates the blocks between
//               folds.  S's hi chain takes all eight k-steps of K_j (both
//               64-dim halves held) before the lo chain's: the accumulator
//               changes once per block.
//   warps 2-17  softmax and folds of O.  Warp w reads TMEM lane quarter w % 4
//               (32 query rows of S, 32 dims of O^T); its part w / 4 - 1 picks
//               32 of a block's keys (softmax) and 32 query columns (folds).
//               softmax of block j: s = S_hi + 2^-11 S_lo (q was scaled by
//               scale * log2(e) before the split), x = s - m_ref of the row;
//               m_ref (the same in the four parts of a row) moves only when a
//               block's maximum exceeds it by more than 8 (lazy rescaling,
//               p = 2^x <= 2^8).  The compute warps exchange one flag per
//               block (shared memory and an mbarrier, waited on with the
//               bounded wait); only when one is raised do they exchange the
//               parts' maxima and move m_ref.  p = 2^x is split into hi/lo
//               fp16 and written to shared memory as P (queries x keys, the B
//               operand of O^T); each part sums p over its keys.
//               fold: O_run += O_hi + 2^-11 O_lo (round to nearest, in
//               registers; times 2^(m_old - m_new) per query when m_ref moved,
//               the factors recomputed from the exchanged maxima), then the
//               O^T chains are zeroed; after every fourth block, before a
//               block whose softmax moved m_ref, and at the end.  Order within
//               block j: read S_j (S_(j+1) may go in), the exchange, p = 2^x
//               and the sums; once O_(j-1) has completed, the P write (O_j may
//               go in once the chains are released), then the fold when due
//               and the release.
//   At the end O = O_run / sum, or the unnormalised partial with its m_ref
//   and sum when the keys are split across CTAs (attn_merge_kernel combines
//   the partials).
// First, the compute warps load the CTA's 128 x 128 fp32 block of Q, scale
// it and split it into the swizzled hi/lo operand tile.  Every wait is
// bounded.
#include "tc_gemm.cuh"

namespace mpg {
namespace {

template <bool kTwoChain>
struct AttnTraits {
  static constexpr int BQ = 128;                 // queries per CTA
  static constexpr int BKEY = kAttnKeyBlock;     // keys per block
  static_assert(BKEY == 128, "the ring's half-block slots and the four 32-key parts assume 128");
  static constexpr int kRing = 5;                // K/V ring slots
  static constexpr int kSlot = 16384;            // one slot: half a K block (64 dims) or half a V block (64 keys)
  // Q: [2 dim halves][256 lines: q_hi of queries 0-127, q_lo of 0-127][128 B], 128-byte swizzle
  static constexpr int kOffQ = 0;
  static constexpr int kOffRing = kOffQ + 2 * 256 * 128;
  // P: [2 key columns: keys 0-63, 64-127][256 lines: p_hi of queries 0-127, p_lo of 0-127][128 B]
  static constexpr int kOffP = kOffRing + kRing * kSlot;
  static constexpr int kOffMax = kOffP + 2 * 256 * 128;         // [2][4 parts][128 rows] maxima
  static constexpr int kOffFlag = kOffMax + 2 * 4 * 128 * 4;     // [2][16 warps] flags
  static constexpr int kOffSum = kOffFlag + 2 * 16 * 4;          // [4 parts][128 rows] sums
  static constexpr int kOffWarp = kOffSum + 4 * 128 * 4;         // [16 warps][32] per-query factors
  static constexpr int kOffBars = kOffWarp + 16 * 32 * 4;
  static constexpr int kNumBars = 2 * kRing + 7 + 1;
  static constexpr int kSmemBytes = 1024 + kOffBars + kNumBars * 8 + 16;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr int kComputeThreads = 512;
  static constexpr int kThreads = 64 + kComputeThreads;
  // TMEM: S at column 0 (lanes = queries; hi chain in columns 0-127, lo in 128-255, one per
  // key), O^T at 256 (lanes = dims; hi 256-383, lo 384-511, one per query)
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColO = 256;
  static constexpr uint32_t kN = kTwoChain ? 256 : 128;   // N of each MMA
  static constexpr int kL = kTwoChain ? 11 : 0;           // lo scale exponent of the split
};

constexpr float kLoScale = 0x1p-11f;
// Lazy rescaling of the online softmax: the reference maximum moves only
// when a block's maximum exceeds it by more than kLazyLog2, so p <= 2^8.
constexpr float kLazyLog2 = 8.0f;
// Blocks of products the O chains accumulate in TMEM between folds into the
// fp32 running output (512 keys: the tensor cores' own accumulation stays
// short, like the split GEMM's K chunks).
constexpr int kFoldBlocks = 4;

// 2^x by the hardware's approximate base-2 exponential (ex2.approx, results
// below 2^-126 flushed to zero: such probabilities add nothing to a sum
// of terms of which the largest is at least 1).
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp32 lanes per instruction (the packed f32x2 forms): d = a * b + c,
// a + b, a - b, a * b, each rounded to nearest like its scalar form.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// p = (p0, p1) split into fp16 hi = RN(p) and lo = RN((p - hi) * 2^L), each
// pair packed into one 32-bit word (the split the operand tiles use).
template <int L>
__device__ __forceinline__ void split2(float p0, float p1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(p0, p1);
  const float2 hb = __half22float2(h);
  float2 r = fsub2(make_float2(p0, p1), hb);
  if constexpr (L == 11) r = fmul2(r, make_float2(2048.0f, 2048.0f));
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// 128-byte swizzled K-major tile (lines of 128 bytes, 8-line groups 1024
// bytes apart), k-step `kk` (16 fp16 = 32 bytes) within one atom column.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t base, int kk) {
  return make_smem_desc(base + (uint32_t)kk * 32u, 16u, 1024u, kSwizzle128B);
}
// 128-byte swizzled MN-major tile: atoms of 64 M/N values x `lines` k-lines
// stored `lines * 128` bytes apart; k-step `kk` covers 16 k-lines.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t base, uint32_t lines, int kk) {
  return make_smem_desc(base + (uint32_t)kk * 2048u, lines * 128u, 1024u, kSwizzle128B);
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int32_t c0, int32_t c1) {
  tma_load_3d(dst, map, bar, c0, c1, 0);
}

template <class T>
__global__ void __launch_bounds__(T::kThreads, 1) attn_kernel(const __grid_constant__ AttnParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem + T::kOffRing;
  float* part_max = reinterpret_cast<float*>(smem + T::kOffMax);
  int* flags = reinterpret_cast<int*>(smem + T::kOffFlag);
  float* part_sum = reinterpret_cast<float*>(smem + T::kOffSum);
  float* warp_vals = reinterpret_cast<float*>(smem + T::kOffWarp);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + T::kOffBars);
  uint64_t* ring_full = bars;
  uint64_t* ring_empty = bars + T::kRing;
  uint64_t* s_full = bars + 2 * T::kRing;
  uint64_t* s_empty = s_full + 1;
  uint64_t* p_full = s_full + 2;
  uint64_t* o_full = s_full + 3;            // O_j complete (which also frees the P^T tile)
  uint64_t* o_empty = s_full + 4;
  uint64_t* q_ready = s_full + 5;
  uint64_t* done_bar = s_full + 6;
  uint64_t* xchg = s_full + 7;              // the compute warps exchange flags, maxima and sums
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(xchg + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qb = blockIdx.x % p.num_q_blk;      // query block
  const int split = blockIdx.x / p.num_q_blk;   // key range
  const int kb0 = split * p.kb_per_split;
  const int kb1 = min(kb0 + p.kb_per_split, (p.lk + T::BKEY - 1) / T::BKEY);
  const int nb = kb1 - kb0;                    // >= 1 (the host never launches an empty range)

  if (threadIdx.x == 0) {
    for (int i = 0; i < T::kRing; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, T::kComputeThreads);
    mbar_init(p_full, T::kComputeThreads);
    mbar_init(o_full, 1);
    mbar_init(o_empty, T::kComputeThreads);
    mbar_init(q_ready, T::kComputeThreads);
    mbar_init(done_bar, 1);
    mbar_init(xchg, T::kComputeThreads);
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

  const uint32_t q_smem = smem_addr(smem + T::kOffQ);
  const uint32_t ring_smem = smem_addr(ring);
  const uint32_t p_smem = smem_addr(smem + T::kOffP);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&p.map_k);
      tma_prefetch_map(&p.map_v);
      uint32_t r = 0;   // ring slots filled so far
      // half `h` of block j: K's dims 64h..64h+63 (all 128 keys), or V's keys
      // 64h..64h+63 (both 64-dim halves)
      auto load = [&](bool is_k, int j, int h) -> bool {
        const uint32_t slot = r % T::kRing;
        if (!mbar_wait(&ring_empty[slot], ((r / T::kRing) & 1u) ^ 1u, ctl)) return false;
        uint8_t* dst = ring + slot * T::kSlot;
        const int key0 = (kb0 + j) * T::BKEY;
        mbar_arrive_expect_tx(&ring_full[slot], T::kSlot);
        if (is_k) {
          tma_load_2d(dst, &p.map_k, &ring_full[slot], 64 * h, key0);
        } else {
          tma_load_2d(dst, &p.map_v, &ring_full[slot], 0, key0 + 64 * h);
          tma_load_2d(dst + T::kSlot / 2, &p.map_v, &ring_full[slot], 64, key0 + 64 * h);
        }
        ++r;
        return true;
      };
      // K_0 first; the rest of the ring only once Q is in (the first S
      // product needs Q and K_0, and every CTA loads them at once)
      bool ok = load(true, 0, 0) && load(true, 0, 1) && mbar_wait(q_ready, 0, ctl);
      for (int j = 0; j < nb && ok; ++j) {
        if (j + 1 < nb) ok = load(true, j + 1, 0) && load(true, j + 1, 1);
        if (ok) ok = load(false, j, 0) && load(false, j, 1);
      }
      // copies issued must land before the CTA may exit
      for (uint32_t i = r > (uint32_t)T::kRing ? r - T::kRing : 0u; i < r; ++i)
        drain_wait(&ring_full[i % T::kRing], (i / T::kRing) & 1u, p.wait_limit_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_s = make_idesc(0u, false, false, 128, 128);     // Q K-major, K K-major
      const uint32_t idesc_o = make_idesc(0u, true, false, 128, T::kN);    // V^T MN-major, P K-major
      const uint32_t t_s = tmem_base + T::kColS, t_o = tmem_base + T::kColO;
      uint32_t r = 0;   // ring slots consumed so far (the producer's order)
      bool ok = mbar_wait(q_ready, 0, ctl);
      tc_fence_after_sync();
      auto take_slot = [&](uint32_t& base) -> bool {
        const uint32_t slot = r % T::kRing;
        if (!mbar_wait(&ring_full[slot], (r / T::kRing) & 1u, ctl)) return false;
        tc_fence_after_sync();
        base = ring_smem + slot * T::kSlot;
        return true;
      };
      auto release_slot = [&]() {
        mma_commit(&ring_empty[r % T::kRing]);
        ++r;
      };
      // S_j = [Q_hi ; Q_lo] K_j^T: the hi chain in columns 0-127, the lo chain
      // in 128-255 (one chain: both into 0-127); per 64-dim half of K_j, the
      // hi chain's four k-steps, then the lo chain's
      auto issue_s = [&](int j) -> bool {
        if (!mbar_wait(s_empty, (j & 1u) ^ 1u, ctl)) return false;
        // both 64-dim halves of K_j, then each chain's eight k-steps in turn
        uint32_t kt[2];
        for (int h = 0; h < 2; ++h) {
          const uint32_t q = r + (uint32_t)h;
          if (!mbar_wait(&ring_full[q % T::kRing], (q / T::kRing) & 1u, ctl)) return false;
          kt[h] = ring_smem + (q % T::kRing) * T::kSlot;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f16(t_s, kmajor_desc(q_smem + (uint32_t)h * 32768u, kk), kmajor_desc(kt[h], kk), idesc_s,
                    (h > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t aq = kmajor_desc(q_smem + (uint32_t)h * 32768u + 16384u, kk);   // Q_lo
            if constexpr (T::kL == 11) {
              mma_f16(t_s + 128u, aq, kmajor_desc(kt[h], kk), idesc_s, (h > 0 || kk > 0) ? 1u : 0u);
            } else {
              mma_f16(t_s, aq, kmajor_desc(kt[h], kk), idesc_s, 1u);
            }
          }
        release_slot();
        release_slot();
        mma_commit(s_full);
        return true;
      };
      // O^T_j (+)= V_j^T [P_hi ; P_lo]^T: A = V^T (dims x keys, MN-major),
      // B = P (256 lines: hi of queries 0-127, lo of 0-127; K-major)
      auto issue_o = [&](int j) -> bool {
        if (!mbar_wait(p_full, j & 1u, ctl)) return false;
        if (!mbar_wait(o_empty, (j & 1u) ^ 1u, ctl)) return false;
        tc_fence_after_sync();
        for (int h = 0; h < 2; ++h) {
          uint32_t vt;
          if (!take_slot(vt)) return false;
          const uint32_t pc = p_smem + (uint32_t)h * 32768u;   // keys 64h..64h+63 of P
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t a = mnmajor_desc(vt, 64, kk);
            // the chains restart after a fold zeroed them (j = 0: nothing to keep)
            const uint32_t acc = (j > 0 || h > 0 || kk > 0) ? 1u : 0u;
            if constexpr (T::kL == 11) {
              mma_f16(t_o, a, kmajor_desc(pc, kk), idesc_o, acc);
            } else {
              mma_f16(t_o, a, kmajor_desc(pc, kk), idesc_o, acc);
              mma_f16(t_o, a, kmajor_desc(pc + 16384u, kk), idesc_o, 1u);
            }
          }
          release_slot();
        }
        mma_commit(o_full);
        return true;
      };
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
      // 128 rows: compute warp w takes rows 8w..8w+7, one row per load (lane
      // l: dims 4l..4l+3, so that a warp reads the row's 512 bytes at once)
      const int w0 = warp - 2;
      float4 xq[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t grow = (int64_t)qb * T::BQ + 8 * w0 + i;
        const float* src = p.q + grow * p.ldq + 4 * lane;
        if (grow < p.lq) {
          if (p.q_vec_ok) {
            xq[i] = __ldg(reinterpret_cast<const float4*>(src));
          } else {
            xq[i] = make_float4(__ldg(src), __ldg(src + 1), __ldg(src + 2), __ldg(src + 3));
          }
        } else {
          xq[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t row = (uint32_t)(8 * w0 + i);
        // q * scale * log2(e), split: the scores come out in base-2 units
        uint32_t h0, l0, h1, l1;
        split_pair(xq[i].x, xq[i].y, p.scale_log2, T::kL == 11 ? 2048.0f : 1.0f, h0, l0);
        split_pair(xq[i].z, xq[i].w, p.scale_log2, T::kL == 11 ? 2048.0f : 1.0f, h1, l1);
        // dims 4l..4l+3: dim half l / 16, 8-byte half (l & 1) of chunk (l / 2) % 8
        // of line `row` (hi) and `128 + row` (lo)
        const uint32_t addr = q_smem + (uint32_t)(lane >> 4) * 32768u +
                              swz_chunk_offset<128>(row, (uint32_t)((lane >> 1) & 7)) + (uint32_t)(lane & 1) * 8u;
        st_shared_v2(addr, h0, h1);
        st_shared_v2(addr + 16384u, l0, l1);
      }
      fence_proxy_async_smem();
      mbar_arrive(q_ready);
    }
    const int cw = warp - 2;
    const int q4 = warp & 3;                      // TMEM lane quarter: query rows (S), dims (O^T) 32*q4..
    const int part = cw >> 2;                     // S: keys 32*part.. of each block; O^T: queries 32*part..
    const uint32_t lane_off = static_cast<uint32_t>(32 * q4) << 16;
    const int row = 32 * q4 + lane;               // this thread's query row of S
    float* f_w = warp_vals + cw * 32;             // per-query factors of this warp's O^T columns
    float o[32];   // O_run of dim 32*q4 + lane for queries 32*part.., relative to m_ref
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i] = 0.0f;
    // the row's reference maximum (base 2; the four parts of a row hold the
    // same) and this part's sum; the first block always sets the reference
    float m_row = 0.0f, l_row = 0.0f;
    uint32_t nx = 0;   // exchanges of the compute warps so far
    bool ok = true;
    // Fold of the O^T chains into the registers: the chains hold the blocks
    // since the last fold, relative to the m_ref before the current block.
    // They are added (hi and lo summed in fp32) and, when the current block
    // moved m_ref, registers and chains are scaled by 2^(m_old - m_new) per
    // query (f_w); `zero` restarts the chains for the next block's products.
    auto fold = [&](bool moved, bool zero) {
      tc_fence_after_sync();
      const uint32_t to = tmem_base + lane_off + T::kColO + 32u * part;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float a[16];
        tmem_ld_16cols(to + 16 * c, a);
        if constexpr (T::kL == 11) {
          float b[16];
          tmem_ld_16cols(to + 128 + 16 * c, b);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 d = ffma2(make_float2(b[i], b[i + 1]), make_float2(kLoScale, kLoScale),
                                   make_float2(a[i], a[i + 1]));
            a[i] = d.x;
            a[i + 1] = d.y;
          }
        } else {
          tmem_ld_wait();
        }
        if (moved) {
#pragma unroll
          for (int i = 0; i < 16; i += 4) {
            const float4 f = reinterpret_cast<const float4*>(f_w)[(16 * c + i) / 4];
            o[16 * c + i] = (o[16 * c + i] + a[i]) * f.x;
            o[16 * c + i + 1] = (o[16 * c + i + 1] + a[i + 1]) * f.y;
            o[16 * c + i + 2] = (o[16 * c + i + 2] + a[i + 2]) * f.z;
            o[16 * c + i + 3] = (o[16 * c + i + 3] + a[i + 3]) * f.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 d = fadd2(make_float2(o[16 * c + i], o[16 * c + i + 1]), make_float2(a[i], a[i + 1]));
            o[16 * c + i] = d.x;
            o[16 * c + i + 1] = d.y;
          }
        }
      }
      if (zero) {
        float z[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) z[i] = 0.0f;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          tmem_st_16cols(to + 16 * c, z);
          if constexpr (T::kL == 11) tmem_st_16cols(to + 128 + 16 * c, z);
        }
        tmem_st_wait();
      }
    };
    // Block j: read this part of the row's S_j (S_(j+1) may then go in),
    // x = s - m_ref, the compute warps' agreement on m_ref, p = 2^x; once
    // O_(j-1) has completed (which also frees the P tile), the fold when it
    // is due and the release of the O^T chains; then P_j, which lets O_j go
    // in; then the row's sum, while O_j runs.
    for (int j = 0; j < nb && ok; ++j) {
      if (!warp_wait(s_full, j & 1u, ctl)) { ok = false; break; }
      tc_fence_after_sync();
      float x[32];
      const uint32_t ts = tmem_base + lane_off + T::kColS + 32u * part;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float a[16];
        tmem_ld_16cols(ts + 16 * h, a);
        if constexpr (T::kL == 11) {
          float b[16];
          tmem_ld_16cols(ts + 128 + 16 * h, b);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 d = ffma2(make_float2(b[i], b[i + 1]), make_float2(kLoScale, kLoScale),
                                   make_float2(a[i], a[i + 1]));
            x[16 * h + i] = d.x;
            x[16 * h + i + 1] = d.y;
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) x[16 * h + i] = a[i];
        }
      }
      tc_fence_before_sync();
      mbar_arrive(s_empty);
      // keys past the end of the sequence score -inf (the same keys in every lane)
      const int key0 = (kb0 + j) * T::BKEY + 32 * part;
      if (key0 + 32 > p.lk) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (key0 + i >= p.lk) x[i] = -INFINITY;
      }
      // x = s - m_ref and its maximum over this part of the row
      float xm = -INFINITY;
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const float2 d = fsub2(make_float2(x[i], x[i + 1]), make_float2(m_row, m_row));
        x[i] = d.x;
        x[i + 1] = d.y;
        xm = fmax3(xm, d.x, d.y);
      }
      // all compute warps agree whether any row needs a new reference
      const bool raise = (j == 0) || __any_sync(0xffffffffu, xm > kLazyLog2);
      int* fl = flags + (nx & 1u) * 16;
      if (lane == 0) fl[cw] = raise ? 1 : 0;
      mbar_arrive(xchg);
      if (!warp_wait(xchg, nx & 1u, ctl)) { ok = false; break; }
      ++nx;
      const int4 f0 = reinterpret_cast<const int4*>(fl)[0], f1 = reinterpret_cast<const int4*>(fl)[1];
      const int4 f2 = reinterpret_cast<const int4*>(fl)[2], f3 = reinterpret_cast<const int4*>(fl)[3];
      const bool moved = ((f0.x | f0.y | f0.z | f0.w) | (f1.x | f1.y | f1.z | f1.w) | (f2.x | f2.y | f2.z | f2.w) |
                          (f3.x | f3.y | f3.z | f3.w)) != 0;   // the same in every compute warp
      const float* pm = part_max + (nx & 1u) * 512;   // [part][row] maxima of x, when moved
      if (moved) {
        part_max[(nx & 1u) * 512 + part * 128 + row] = xm;
        mbar_arrive(xchg);
        if (!warp_wait(xchg, nx & 1u, ctl)) { ok = false; break; }
        ++nx;
        const float mb = fmaxf(fmaxf(pm[row], pm[128 + row]), fmaxf(pm[256 + row], pm[384 + row]));
        const bool mv = (j == 0) || mb > kLazyLog2;
        const float dm = mv ? mb : 0.0f;
        m_row += dm;
        // 2^(m_old - m_new); nothing is kept before the first block
        l_row *= (j == 0) ? 0.0f : (mv ? exp2_approx(-mb) : 1.0f);
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 d = fsub2(make_float2(x[i], x[i + 1]), make_float2(dm, dm));
          x[i] = d.x;
          x[i + 1] = d.y;
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) x[i] = exp2_approx(x[i]);
      // this part's sum of p over the row's keys
      {
        float2 s0 = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          s0 = fadd2(s0, make_float2(x[i], x[i + 1]));
          s1 = fadd2(s1, make_float2(x[i + 2], x[i + 3]));
        }
        l_row += (s0.x + s0.y) + (s1.x + s1.y);
      }
      // O_(j-1) has completed: the P tile is free and the O^T chains hold
      // every block up to j-1
      if (j >= 1 && !warp_wait(o_full, (j - 1) & 1u, ctl)) { ok = false; break; }
      // P, the K-major B operand of O^T: line `row` (hi) and 128 + row (lo)
      // of key column part / 2, this part's 32 keys as 4 chunks of 8
      {
        const uint32_t line = p_smem + (uint32_t)(part >> 1) * 32768u + (uint32_t)row * 128u;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t h[4], l[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) split2<T::kL>(x[8 * c + 2 * e], x[8 * c + 2 * e + 1], h[e], l[e]);
          const uint32_t off = (((uint32_t)((part & 1) * 4 + c)) ^ ((uint32_t)row & 7u)) << 4;
          st_shared_v4(line + off, h[0], h[1], h[2], h[3]);
          st_shared_v4(line + 16384u + off, l[0], l[1], l[2], l[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(p_full);
      if (j >= 1) {
        // fold after every kFoldBlocks blocks and before products relative
        // to a moved m_ref, then release the chains (O_j waits for both)
        if (moved || j % kFoldBlocks == 0) {
          if (moved) {
            // the factors of this warp's query columns, from the exchanged maxima
            const int qc = 32 * part + lane;
            const float mq = fmaxf(fmaxf(pm[qc], pm[128 + qc]), fmaxf(pm[256 + qc], pm[384 + qc]));
            f_w[lane] = mq > kLazyLog2 ? exp2_approx(-mq) : 1.0f;
            __syncwarp();
          }
          fold(moved, true);
        }
        tc_fence_before_sync();
        mbar_arrive(o_empty);
      }
    }
    // the last fold, once the last block's products have completed
    if (ok) {
      ok = warp_wait(o_full, (nb - 1) & 1u, ctl);
      if (ok) fold(false, false);
    }
    // the row's sum is the sum of its four parts' sums
    if (ok) {
      part_sum[part * 128 + row] = l_row;
      mbar_arrive(xchg);
      ok = warp_wait(xchg, nx & 1u, ctl);
      ++nx;
    }
    if (ok) {
      const int64_t q0 = (int64_t)qb * T::BQ + 32 * part;   // this warp's output queries
      const int dim = 32 * q4 + lane;
      const int qc = 32 * part + lane;
      const float lq_sum = (part_sum[qc] + part_sum[128 + qc]) + (part_sum[256 + qc] + part_sum[384 + qc]);
      if (p.splits == 1) {
        f_w[lane] = 1.0f / lq_sum;
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          const float4 f = reinterpret_cast<const float4*>(f_w)[i / 4];
          const float fs[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            if (q0 + i + e < p.lq) p.o[(q0 + i + e) * p.ldo + dim] = o[i + e] * fs[e];
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (q0 + i < p.lq) p.part_o[((int64_t)split * p.lq + q0 + i) * 128 + dim] = o[i];
        const int64_t grow = (int64_t)qb * T::BQ + row;
        if (part == 0 && grow < p.lq) {
          const float l_all = (part_sum[row] + part_sum[128 + row]) + (part_sum[256 + row] + part_sum[384 + row]);
          p.part_m[(int64_t)split * p.lq + grow] = m_row;
          p.part_l[(int64_t)split * p.lq + grow] = l_all;
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

int attention_smem_bytes() { return AttnTraits<true>::kSmemBytes; }

cudaError_t launch_attention(const AttnParams& p, bool two_chain, cudaStream_t stream) {
  cudaError_t e = two_chain ? launch_kernel<AttnTraits<true>>(p, stream)
                            : launch_kernel<AttnTraits<false>>(p, stream);
  if (e != cudaSuccess || p.splits == 1) return e;
  const int64_t items = (int64_t)p.lq * 32;
  attn_merge_kernel<<<(unsigned)((items + 255) / 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mpg
