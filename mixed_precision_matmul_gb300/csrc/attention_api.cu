// mpg_attention: argument checks, the division of the keys among CTAs and
// the workspace of their partial results, tensor maps of K and V, launch of
// the fused kernel (csrc/attention.cu) and of the merge.
#include <cmath>
#include <cstring>

#include "host.h"

using namespace mpg;

namespace {

// --------------------------------------------------------------------------
// fused attention: key ranges and workspace
// --------------------------------------------------------------------------
struct AttnSplit {
  int splits = 1, kb_per_split = 1;
  size_t off_m = 0, off_l = 0, bytes = 0;
};

AttnSplit attention_split(int64_t lq, int64_t lk, int32_t key_splits, int sm_count) {
  AttnSplit a;
  const int64_t nkb = (lk + kAttnKeyBlock - 1) / kAttnKeyBlock;
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
  s = encode_map(&p.map_k, Kop, d, lk, 1, 64, kAttnKeyBlock);
  if (s != MPG_OK) return s;
  s = encode_map(&p.map_v, Vop, d, lk, 1, 64, kAttnKeyBlock / 2);
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
