// mpg_gemm_host: the product on A, B and C in host memory.  Packed device
// copies (lines padded to 16 bytes) in the caller's workspace; B first, then
// row chunks of A and C (whole matrices when batch > 1) pipelined on two
// internal copy streams against the product on the caller's stream.
#include <algorithm>

#include "host.h"

using namespace mpg;

namespace {

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
  static std::mutex streams_mu;
  std::lock_guard<std::mutex> lock(streams_mu);
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

}  // namespace

extern "C" {

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

}  // extern "C"
