// Hardware check of the tcgen05 accumulator map: one CTA runs one k-block
// (K = 64, four K = 16 instructions) of the one-CTA product's MMA path on
// operands it writes into 128-byte swizzled shared memory with the product
// kernels' own layout code and descriptors, then every warp copies out the
// raw registers of tcgen05.ld.32x32b.x32, unscattered, so that the host can
// place them with mpg_tmem_acc_coords and compare with its own product.
// (The mma.sync counterpart is "feat(cuda-device): derive the m16n8k16
// accumulator fragment layout", section "Verified against hardware".)
#include "tc_gemm.cuh"

namespace mpg {
namespace {

// The direct 16-bit path's traits: 128-byte K-major lines of 64 fp16 values,
// K = 16 per instruction.
using ProbeT = TcTraits<Src::kTmaDirect, Conv::kNone, Op::kF16, SrcT::kF16, 128>;
constexpr int kProbeK = 64;
constexpr int kProbeMaxN = 256;
constexpr int kProbeSmem = 1024 + 128 * 128 + kProbeMaxN * 128 + 64;

__global__ void __launch_bounds__(128, 1) probe_tmem_kernel(const uint16_t* __restrict__ A,
                                                             const uint16_t* __restrict__ B, int n,
                                                             float* __restrict__ D, uint32_t* status,
                                                             uint64_t limit_ns) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a_tile = smem;                       // 128 lines of 128 bytes
  uint8_t* b_tile = smem + 128 * 128;           // n lines of 128 bytes
  uint64_t* bar = reinterpret_cast<uint64_t*>(b_tile + kProbeMaxN * 128);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // operands: line r of a tile is row r of A (resp. column r of B), its
  // 16-byte chunk c holds k = 8c .. 8c+7, placed by the 128-byte swizzle
  const uint32_t a_addr = smem_addr(a_tile), b_addr = smem_addr(b_tile);
  for (int i = threadIdx.x; i < (128 + n) * 8; i += blockDim.x) {
    const bool isA = i < 128 * 8;
    const int w = isA ? i : i - 128 * 8;
    const int line = w >> 3, ch = w & 7;
    const uint4 v = *reinterpret_cast<const uint4*>((isA ? A : B) + line * kProbeK + ch * 8);
    st_shared_v4((isA ? a_addr : b_addr) + swz_chunk_offset<128>(line, ch), v.x, v.y, v.z, v.w);
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  const uint32_t ncols = n <= 32 ? 32 : n <= 64 ? 64 : n <= 128 ? 128 : 256;
  if (warp == 0) {
    tmem_alloc(tmem_slot, ncols);
    tmem_relinquish();
    tc_fence_before_sync();
  }
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  WaitCtl ctl;
  ctl.abort = abort_flag;
  ctl.status = status;
  ctl.limit_ns = limit_ns;

  if (threadIdx.x == 0) {
    const uint32_t idesc = make_idesc(0u /* f16 */, false, false, 128, (uint32_t)n);
#pragma unroll
    for (int ks = 0; ks < ProbeT::kKSteps; ++ks)
      mma_f16(tmem_base, operand_desc<ProbeT>(a_addr, false, ks), operand_desc<ProbeT>(b_addr, false, ks), idesc,
              ks > 0 ? 1u : 0u);
    mma_commit(bar);
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
      float* out = D + ((size_t)(warp * 32 + lane) * (n / 32) + c) * 32;
#pragma unroll
      for (int r = 0; r < 32; ++r) out[r] = v[r];
    }
  } else {
    // the MMAs may still run: let them finish before TMEM is released
    drain_wait(bar, 0, limit_ns);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, ncols);
  }
}

}  // namespace

cudaError_t launch_probe_tmem(const void* a, const void* b, int n, float* d, uint32_t* status, uint64_t limit_ns,
                              cudaStream_t stream) {
  if (n != 64 && n != 128 && n != 256) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(probe_tmem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
  if (e != cudaSuccess) return e;
  probe_tmem_kernel<<<1, 128, kProbeSmem, stream>>>(static_cast<const uint16_t*>(a), static_cast<const uint16_t*>(b),
                                                     n, d, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace mpg
