// Host-side common services of the C ABI: error messages, the per-device
// cache (SM count, shared-memory limit, status word, the tensor-map encoder)
// and TMA tensor-map encoding.
#include <cstdarg>
#include <cstdio>

#include "host.h"

namespace mpg {

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

DeviceInfo g_devices[kMaxDevices];

namespace {
std::mutex g_dev_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
}  // namespace

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
  std::lock_guard<std::mutex> lock(g_dev_mu);
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

bool tma_ok(const Operand& x, int64_t batch) {
  const int64_t es = elem_bytes(x.dt);
  if (reinterpret_cast<uintptr_t>(x.ptr) % 16 != 0) return false;
  if ((x.ld * es) % 16 != 0 || x.ld * es >= (int64_t(1) << 40)) return false;
  if (batch > 1 && ((x.stride * es) % 16 != 0 || x.stride * es >= (int64_t(1) << 40))) return false;
  return true;
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

}  // namespace mpg
