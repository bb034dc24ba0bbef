"""mixed_precision_matmul_gb300 — Python binding of the ``libmpgemm`` C ABI.

Argument marshalling only: every step of the product runs in the library's
CUDA kernels.  PyTorch supplies device memory, the current stream and tensor
metadata (pointers, strides).  There is no fallback: if the CUDA library is not
built, importing the compute entry points raises.

Entry points mirror ``include/mpgemm.h``:

* :func:`gemm`   C = alpha*A*B + beta*C on torch tensors (layouts read from
  strides: a 2-D operand with unit column stride is row-major, with unit row
  stride column-major; a leading batch dimension gives the batch stride).
* :func:`gemm_raw`   the plain-pointer form of ``mpg_gemm_ex``.
* :func:`acc_coords`, :func:`acc_offset`, :func:`acc_matrix_offset`,
  :func:`acc_decode`, :func:`tmem_acc_coords`, :func:`tmem_acc_decode`   host decode of accumulator
  fragments.
* :func:`probe_mma_m16n8k16`, :func:`selftest_wait_timeout`,
  :func:`device_status`.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import _build

# precision modes (mpg_precision)
(FP16_F32ACC, BF16_F32ACC, TF32, SPLIT_FP16_3CHAIN, SPLIT_FP16_1CHAIN, FP32_FFMA, SPLIT_A_FP16_2CHAIN,
 SPLIT_FP16_4CHAIN) = range(8)
MODE_NAMES = {
    "fp16": FP16_F32ACC, "bf16": BF16_F32ACC, "tf32": TF32,
    "split3": SPLIT_FP16_3CHAIN, "split1": SPLIT_FP16_1CHAIN, "ffma": FP32_FFMA,
    "split2a": SPLIT_A_FP16_2CHAIN, "split4": SPLIT_FP16_4CHAIN,
}
# storage types (mpg_dtype) and layouts (mpg_layout)
F32, F16, BF16 = 0, 1, 2
ROW_MAJOR, COL_MAJOR = 0, 1
# status codes (mpg_status)
STATUS = {0: "MPG_OK", 1: "MPG_ERR_INVALID_ARG", 2: "MPG_ERR_UNSUPPORTED", 3: "MPG_ERR_NO_DEVICE",
          4: "MPG_ERR_WORKSPACE", 5: "MPG_ERR_CUDA", 6: "MPG_ERR_TIMEOUT"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_NO_DEVICE, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(7)

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mpgemm.h")


class MpgError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class Options(ctypes.Structure):
    _fields_ = [
        ("split_exp_a", ctypes.c_int32),
        ("split_exp_b", ctypes.c_int32),
        ("splitk", ctypes.c_int32),
        ("force_generic_load", ctypes.c_int32),
        ("tile_n", ctypes.c_int32),
        ("wait_timeout_ns", ctypes.c_int64),
        ("split_chunk_k", ctypes.c_int32),
        ("prepass", ctypes.c_int32),
        ("c_dtype", ctypes.c_int32),
        ("cta_pair", ctypes.c_int32),
        ("tail_split", ctypes.c_int32),
        ("split_plain_lo", ctypes.c_int32),
        ("split_lo_shared", ctypes.c_int32),
        ("reserved", ctypes.c_int32 * 1),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def build(force: bool = False) -> str:
    return _build.build(force=force)


def lib():
    """The loaded libmpgemm (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_build.LIB):
            raise ImportError(
                f"libmpgemm.so is not built ({_build.LIB}); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(_build.LIB)
        i64, i32, f32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
        gemm_args = [i64, i64, i64, i64,
                     vp, i64, i64, i32, i32,
                     vp, i64, i64, i32, i32,
                     vp, i64, i64, f32, f32, i32, vp, sz, vp]
        L.mpg_gemm.argtypes = gemm_args
        L.mpg_gemm.restype = i32
        L.mpg_gemm_ex.argtypes = gemm_args + [ctypes.POINTER(Options)]
        L.mpg_gemm_ex.restype = i32
        L.mpg_gemm_noalloc.argtypes = gemm_args[:20] + [vp, ctypes.POINTER(Options)]
        L.mpg_gemm_noalloc.restype = i32
        L.mpg_gemm_workspace_size.argtypes = [i64, i64, i64, i64, i32, ctypes.POINTER(Options)]
        L.mpg_gemm_workspace_size.restype = sz
        L.mpg_gemm_workspace_size_ex.argtypes = [i64, i64, i64, i64, vp, i64, i64, i32, i32, vp, i64, i64, i32, i32,
                                                 i32, ctypes.POINTER(Options)]
        L.mpg_gemm_workspace_size_ex.restype = sz
        L.mpg_attention_workspace_size.argtypes = [i64, i64, i64, i32]
        L.mpg_attention_workspace_size.restype = sz
        L.mpg_attention.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, f32, i32, i32, vp, sz, vp]
        L.mpg_attention.restype = i32
        L.mpg_gemm_host.argtypes = gemm_args + [ctypes.POINTER(Options)]
        L.mpg_gemm_host.restype = i32
        L.mpg_gemm_host_workspace_size.argtypes = [i64, i64, i64, i64, i64, i64, i32, i32, i64, i64, i32, i32,
                                                   i64, i64, f32, f32, i32, ctypes.POINTER(Options)]
        L.mpg_gemm_host_workspace_size.restype = sz
        L.mpg_options_init.argtypes = [ctypes.POINTER(Options)]
        L.mpg_options_init.restype = None
        L.mpg_device_status.argtypes = [vp]
        L.mpg_device_status.restype = i32
        L.mpg_last_error_string.argtypes = []
        L.mpg_last_error_string.restype = ctypes.c_char_p
        L.mpg_version.argtypes = []
        L.mpg_version.restype = i32
        pi = ctypes.POINTER(ctypes.c_int)
        L.mpg_acc_coords.argtypes = [i32, i32, pi, pi]
        L.mpg_acc_coords.restype = i32
        L.mpg_acc_offset.argtypes = [i32, i32]
        L.mpg_acc_offset.restype = i32
        L.mpg_acc_matrix_offset.argtypes = [i32, i32, i64, i64, i64, i64]
        L.mpg_acc_matrix_offset.restype = i64
        L.mpg_acc_decode.argtypes = [i32, pi, pi]
        L.mpg_acc_decode.restype = i32
        L.mpg_tmem_acc_coords.argtypes = [i32, i32, i32, i32, i32, i32, pi, pi]
        L.mpg_tmem_acc_coords.restype = i32
        L.mpg_tmem_acc_decode.argtypes = [i32, i32, i32, i32, pi, pi, pi, pi, pi]
        L.mpg_tmem_acc_decode.restype = i32
        L.mpg_probe_tmem_acc.argtypes = [vp, vp, i32, vp, vp]
        L.mpg_probe_tmem_acc.restype = i32
        L.mpg_probe_tmem_acc_pair.argtypes = [vp, vp, i32, vp, vp]
        L.mpg_probe_tmem_acc_pair.restype = i32
        L.mpg_probe_fma_rate.argtypes = [vp, ctypes.c_int64, i32, i32, vp]
        L.mpg_probe_fma_rate.restype = i32
        L.mpg_probe_mma_m16n8k16.argtypes = [vp, vp, vp, vp]
        L.mpg_probe_mma_m16n8k16.restype = i32
        for nm in ("mpg_frag_a_coords", "mpg_frag_a_decode", "mpg_frag_b_coords", "mpg_frag_b_decode"):
            getattr(L, nm).argtypes = [i32, i32, pi, pi]
            getattr(L, nm).restype = i32
        L.mpg_probe_mma_m16n8k16_fragments.argtypes = [vp, vp, vp, vp]
        L.mpg_probe_mma_m16n8k16_fragments.restype = i32
        L.mpg_probe_epilogue_staging.argtypes = [vp, vp, ctypes.c_int64, i32, vp]
        L.mpg_probe_epilogue_staging.restype = i32
        L.mpg_selftest_wait_timeout.argtypes = [i64, vp]
        L.mpg_selftest_wait_timeout.restype = i32
        _lib = L
        return L


def header_functions() -> list[str]:
    """Names of the functions include/mpgemm.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return sorted(set(re.findall(r"\b(mpg_[a-z0-9_]+)\s*\(", text)))


def last_error() -> str:
    s = lib().mpg_last_error_string()
    return s.decode() if s else ""


def _check(status: int):
    if status != OK:
        raise MpgError(status, last_error())


def options(**kw) -> Options:
    o = Options()
    lib().mpg_options_init(ctypes.byref(o))
    for k, v in kw.items():
        setattr(o, k, v)
    return o


# ---------------------------------------------------------------------------
# raw C-ABI form
# ---------------------------------------------------------------------------

def gemm_raw(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype, b_layout,
             C, ldc, strideC, alpha, beta, mode, workspace=0, workspace_bytes=0, stream=0,
             opts: Options | None = None, check: bool = True) -> int:
    """mpg_gemm_ex with integer device pointers; returns the status code
    (raises MpgError on failure when ``check``)."""
    st = lib().mpg_gemm_ex(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype,
                           b_layout, C, ldc, strideC, float(alpha), float(beta), mode, workspace or None,
                           workspace_bytes, stream or None, ctypes.byref(opts) if opts is not None else None)
    if check:
        _check(st)
    return st


def gemm_noalloc_raw(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype,
                     b_layout, C, ldc, strideC, alpha, beta, mode, stream=0,
                     opts: Options | None = None, check: bool = True) -> int:
    """mpg_gemm_noalloc: the product without a workspace argument, for callers
    that cannot allocate device memory (split-K partial sums go to the
    library's fixed 16 MiB static scratch; larger needs are rejected)."""
    st = lib().mpg_gemm_noalloc(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype,
                                b_layout, C, ldc, strideC, float(alpha), float(beta), mode, stream or None,
                                ctypes.byref(opts) if opts is not None else None)
    if check:
        _check(st)
    return st


def gemm_host_raw(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype, b_layout,
                  C, ldc, strideC, alpha, beta, mode, workspace, workspace_bytes, stream=0,
                  opts: Options | None = None, check: bool = True) -> int:
    """mpg_gemm_host: A, B and C are HOST addresses; the call copies in,
    multiplies and copies C back, enqueued on `stream` (device workspace of
    host_workspace_size() bytes)."""
    st = lib().mpg_gemm_host(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype,
                             b_layout, C, ldc, strideC, float(alpha), float(beta), mode, workspace or None,
                             workspace_bytes, stream or None, ctypes.byref(opts) if opts is not None else None)
    if check:
        _check(st)
    return st


def host_workspace_size(m, n, k, batch, lda, strideA, a_dtype, a_layout, ldb, strideB, b_dtype, b_layout,
                        ldc, strideC, alpha, beta, mode, opts: Options | None = None) -> int:
    return int(lib().mpg_gemm_host_workspace_size(m, n, k, batch, lda, strideA, a_dtype, a_layout, ldb, strideB,
                                                  b_dtype, b_layout, ldc, strideC, float(alpha), float(beta), mode,
                                                  ctypes.byref(opts) if opts is not None else None))


ATTN_SPLIT_2CHAIN = 0
ATTN_SPLIT_1CHAIN = 1


def attention_workspace_size(lq, lk, d=128, key_splits=0) -> int:
    return int(lib().mpg_attention_workspace_size(lq, lk, d, key_splits))


def attention_raw(lq, lk, d, Q, ldq, K, ldk, V, ldv, O, ldo, scale, mode=ATTN_SPLIT_2CHAIN, key_splits=0,
                  workspace=0, workspace_bytes=0, stream=0, check: bool = True) -> int:
    """mpg_attention on device addresses: O = softmax(scale * Q K^T) V with Q
    fp32 and K, V fp16 (lq x d, lk x d, lk x d row-major)."""
    st = lib().mpg_attention(lq, lk, d, Q, ldq, K, ldk, V, ldv, O, ldo, float(scale), mode, key_splits,
                             workspace or None, workspace_bytes, stream or None)
    if check:
        _check(st)
    return st


def attention(Q, K, V, O=None, scale: float | None = None, mode=ATTN_SPLIT_2CHAIN, key_splits=0, stream=None):
    """Fused prompt attention on CUDA tensors: Q (lq x d) fp32, K and V
    (lk x d) fp16, O (lq x d) fp32 (allocated when not given); the scale
    defaults to 1/sqrt(d).  Returns O."""
    torch = _torch()
    lq, d = Q.shape
    lk = K.shape[0]
    if K.shape[1] != d or V.shape != K.shape:
        raise ValueError("attention operand shapes disagree")
    if Q.dtype != torch.float32 or K.dtype != torch.float16 or V.dtype != torch.float16:
        raise ValueError("Q must be fp32, K and V fp16")
    if Q.stride(1) != 1 or K.stride(1) != 1 or V.stride(1) != 1:
        raise ValueError("operands must be row-major with unit column stride")
    if O is None:
        O = torch.empty((lq, d), dtype=torch.float32, device=Q.device)
    if scale is None:
        scale = 1.0 / float(d) ** 0.5
    ws_bytes = attention_workspace_size(lq, lk, d, key_splits)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=Q.device) if ws_bytes else None
    attention_raw(lq, lk, d, Q.data_ptr(), Q.stride(0), K.data_ptr(), K.stride(0), V.data_ptr(), V.stride(0),
                  O.data_ptr(), O.stride(0), scale, mode, key_splits, ws.data_ptr() if ws is not None else 0,
                  ws_bytes, _stream_handle(stream))
    return O


def workspace_size_ex(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb, strideB, b_dtype, b_layout,
                      mode, opts: Options | None = None) -> int:
    """Workspace for this exact call (includes aligned copies of operands
    TMA cannot describe)."""
    return int(lib().mpg_gemm_workspace_size_ex(m, n, k, batch, A, lda, strideA, a_dtype, a_layout, B, ldb,
                                                strideB, b_dtype, b_layout, mode,
                                                ctypes.byref(opts) if opts is not None else None))


def workspace_size(m, n, k, batch, mode, opts: Options | None = None) -> int:
    return int(lib().mpg_gemm_workspace_size(m, n, k, batch, mode,
                                             ctypes.byref(opts) if opts is not None else None))


def device_status(stream=None) -> int:
    return lib().mpg_device_status(_stream_handle(stream))


# ---------------------------------------------------------------------------
# torch form
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(stream):
    if stream is None:
        torch = _torch()
        if not torch.cuda.is_available():
            return None
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _operand(t, rows: int, cols: int):
    """(layout, ld, batch_stride) of a 2-D or batched 3-D operand view."""
    s = t.stride()
    r_st, c_st = s[-2], s[-1]
    bstride = s[0] if t.dim() == 3 else 0
    if c_st == 1 and (r_st >= max(cols, 1) or rows <= 1):
        return ROW_MAJOR, max(r_st, cols, 1), bstride
    if r_st == 1 and (c_st >= max(rows, 1) or cols <= 1):
        return COL_MAJOR, max(c_st, rows, 1), bstride
    raise ValueError(f"operand with strides {s} is neither row- nor column-major")


def gemm(A, B, C, alpha: float = 1.0, beta: float = 0.0, mode=BF16_F32ACC, workspace=None,
         opts: Options | None = None, stream=None):
    """C = alpha * A @ B + beta * C on CUDA tensors, in place on C.

    A is (m, k) or (batch, m, k), B is (k, n) or (batch, k, n), C is fp32,
    fp16 or bf16 (m, n) or (batch, m, n) with unit column stride (a 16-bit C
    gets one final rounding of the fp32 result).  ``mode`` is one of the
    precision constants (or a name from MODE_NAMES).  A workspace for split-K
    is allocated through torch when the library asks for one and none is
    given.  Returns C.
    """
    torch = _torch()
    if isinstance(mode, str):
        mode = MODE_NAMES[mode]
    batched = C.dim() == 3
    batch = C.shape[0] if batched else 1
    m, k = A.shape[-2], A.shape[-1]
    n = B.shape[-1]
    if B.shape[-2] != k or C.shape[-2] != m or C.shape[-1] != n:
        raise ValueError("shape mismatch")
    if C.dtype not in (torch.float32, torch.float16, torch.bfloat16) or C.stride(-1) != 1:
        raise ValueError("C must be fp32, fp16 or bf16 with unit column stride")
    if C.dtype != torch.float32 or opts is not None:
        # the output type always follows C's own dtype
        o = Options()
        if opts is not None:
            ctypes.memmove(ctypes.byref(o), ctypes.byref(opts), ctypes.sizeof(Options))
        else:
            lib().mpg_options_init(ctypes.byref(o))
        o.c_dtype = _dtype_code(C)
        opts = o
    a_layout, lda, sa = _operand(A, m, k)
    b_layout, ldb, sb = _operand(B, k, n)
    ldc = max(C.stride(-2), n, 1)
    sc = C.stride(0) if batched else 0
    ws_bytes = workspace_size_ex(m, n, k, batch, A.data_ptr(), lda, sa, _dtype_code(A), a_layout,
                                 B.data_ptr(), ldb, sb, _dtype_code(B), b_layout, mode, opts)
    if workspace is None and ws_bytes > 0:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=C.device)
    ws_ptr = workspace.data_ptr() if workspace is not None else 0
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    gemm_raw(m, n, k, batch, A.data_ptr(), lda, sa, _dtype_code(A), a_layout,
             B.data_ptr(), ldb, sb, _dtype_code(B), b_layout, C.data_ptr(), ldc, sc,
             alpha, beta, mode, ws_ptr, ws_len, _stream_handle(stream), opts)
    return C


def gemm_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, mode=BF16_F32ACC, opts: Options | None = None,
              device=None, stream=None):
    """C = alpha * A @ B + beta * C on CPU tensors (page-locked ones, e.g.
    from ``tensor.pin_memory()``, let the copies run asynchronously), through
    mpg_gemm_host: the call copies A, B and C to the device, multiplies, and
    copies C back into the same host tensor.  The device workspace is
    allocated through torch on ``device`` (default: the current CUDA device).
    Returns C once the product has completed (the stream is synchronised)."""
    torch = _torch()
    if isinstance(mode, str):
        mode = MODE_NAMES[mode]
    for t in (A, B, C):
        if t.is_cuda:
            raise ValueError("gemm_host takes host (CPU) tensors")
    batched = C.dim() == 3
    batch = C.shape[0] if batched else 1
    m, k = A.shape[-2], A.shape[-1]
    n = B.shape[-1]
    if B.shape[-2] != k or C.shape[-2] != m or C.shape[-1] != n:
        raise ValueError("shape mismatch")
    if C.dtype not in (torch.float32, torch.float16, torch.bfloat16) or C.stride(-1) != 1:
        raise ValueError("C must be fp32, fp16 or bf16 with unit column stride")
    o = Options()
    if opts is not None:
        ctypes.memmove(ctypes.byref(o), ctypes.byref(opts), ctypes.sizeof(Options))
    else:
        lib().mpg_options_init(ctypes.byref(o))
    o.c_dtype = _dtype_code(C)
    a_layout, lda, sa = _operand(A, m, k)
    b_layout, ldb, sb = _operand(B, k, n)
    ldc = max(C.stride(-2), n, 1)
    sc = C.stride(0) if batched else 0
    ws_bytes = host_workspace_size(m, n, k, batch, lda, sa, _dtype_code(A), a_layout, ldb, sb, _dtype_code(B),
                                   b_layout, ldc, sc, alpha, beta, mode, o)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = torch.cuda.current_stream() if stream is None else stream
        gemm_host_raw(m, n, k, batch, A.data_ptr(), lda, sa, _dtype_code(A), a_layout, B.data_ptr(), ldb, sb,
                      _dtype_code(B), b_layout, C.data_ptr(), ldc, sc, alpha, beta, mode, ws.data_ptr(), ws_bytes,
                      st.cuda_stream, o)
        st.synchronize()
    return C


# ---------------------------------------------------------------------------
# accumulator fragment decode (host)
# ---------------------------------------------------------------------------

def acc_coords(lane: int, j: int) -> tuple[int, int] | None:
    r, c = ctypes.c_int(), ctypes.c_int()
    if lib().mpg_acc_coords(lane, j, ctypes.byref(r), ctypes.byref(c)) != 0:
        return None
    return r.value, c.value


def acc_offset(lane: int, j: int) -> int:
    return lib().mpg_acc_offset(lane, j)


def acc_matrix_offset(lane: int, j: int, tile_row: int, tile_col: int, row_stride: int, limit: int):
    v = lib().mpg_acc_matrix_offset(lane, j, tile_row, tile_col, row_stride, limit)
    return None if v < 0 else v


def acc_decode(offset: int) -> tuple[int, int] | None:
    ln, j = ctypes.c_int(), ctypes.c_int()
    if lib().mpg_acc_decode(offset, ctypes.byref(ln), ctypes.byref(j)) != 0:
        return None
    return ln.value, j.value


def tmem_acc_coords(warp: int, lane: int, reg: int, col_base: int = 0, m_shape: int = 128, cta_rank: int = 0):
    """(row, col) of register `reg` of lane `lane` of warp `warp` in a
    tcgen05.ld.32x32b from column `col_base` (mpg_tmem_acc_coords)."""
    r, c = ctypes.c_int(), ctypes.c_int()
    if lib().mpg_tmem_acc_coords(m_shape, cta_rank, warp, lane, reg, col_base, ctypes.byref(r),
                                 ctypes.byref(c)) != 0:
        return None
    return r.value, c.value


def tmem_acc_decode(row: int, col: int, load_cols: int = 32, m_shape: int = 128):
    """(cta_rank, warp, lane, reg, col_base) holding D(row, col) in loads of
    `load_cols` columns (mpg_tmem_acc_decode)."""
    out = [ctypes.c_int() for _ in range(5)]
    if lib().mpg_tmem_acc_decode(m_shape, row, col, load_cols, *[ctypes.byref(x) for x in out]) != 0:
        return None
    return tuple(x.value for x in out)


def _pair(fn, x, y):
    u, v = ctypes.c_int(), ctypes.c_int()
    if fn(x, y, ctypes.byref(u), ctypes.byref(v)) != 0:
        return None
    return u.value, v.value


def frag_a_coords(lane: int, i: int):
    """(row, col) of value i (register i//2, half i%2) of an A fragment."""
    return _pair(lib().mpg_frag_a_coords, lane, i)


def frag_a_decode(row: int, col: int):
    return _pair(lib().mpg_frag_a_decode, row, col)


def frag_b_coords(lane: int, i: int):
    """(k, n) of value i (register i//2, half i%2) of a B fragment."""
    return _pair(lib().mpg_frag_b_coords, lane, i)


def frag_b_decode(k: int, n: int):
    return _pair(lib().mpg_frag_b_decode, k, n)


# ---------------------------------------------------------------------------
# hardware checks
# ---------------------------------------------------------------------------

def probe_mma_m16n8k16(A16, B16, stream=None):
    """One mma.sync m16n8k16 on fp16 A (16x16 row-major) and B (16x8, stored
    column-major, i.e. B.t() contiguous); returns the raw (32, 4) fragments."""
    torch = _torch()
    a = A16.to(torch.float16).contiguous()
    bt = B16.to(torch.float16).t().contiguous()  # column-major storage of B
    d = torch.empty((32, 4), dtype=torch.float32, device=a.device)
    _check(lib().mpg_probe_mma_m16n8k16(a.data_ptr(), bt.data_ptr(), d.data_ptr(), _stream_handle(stream)))
    return d


def probe_mma_m16n8k16_fragments(a_frag, b_frag, stream=None):
    """mma.sync m16n8k16 on fragments given per lane: a_frag (32, 4) and
    b_frag (32, 2) int32 tensors of packed fp16 pairs; returns (32, 4) floats."""
    torch = _torch()
    a = a_frag.to(torch.int32).contiguous()
    b = b_frag.to(torch.int32).contiguous()
    d = torch.empty((32, 4), dtype=torch.float32, device=a.device)
    _check(lib().mpg_probe_mma_m16n8k16_fragments(a.data_ptr(), b.data_ptr(), d.data_ptr(),
                                                   _stream_handle(stream)))
    return d


def probe_tmem_acc(A16, Bt16, stream=None):
    """One k-block (K = 64) of the one-CTA tcgen05 path on fp16 A (128 x 64)
    and B given as Bt (n x 64, row j = column j of B); returns the raw
    tcgen05.ld registers as a (4 warps, 32 lanes, n/32 loads, 32 regs) tensor."""
    torch = _torch()
    a = A16.to(torch.float16).contiguous()
    bt = Bt16.to(torch.float16).contiguous()
    n = bt.shape[0]
    if a.shape != (128, 64) or bt.shape[1] != 64:
        raise ValueError("A must be 128 x 64 and Bt n x 64")
    d = torch.empty((4, 32, n // 32, 32), dtype=torch.float32, device=a.device)
    _check(lib().mpg_probe_tmem_acc(a.data_ptr(), bt.data_ptr(), n, d.data_ptr(), _stream_handle(stream)))
    return d


def probe_fma_rate(blocks, iters, packed=True, out=None, stream=None):
    """mpg_probe_fma_rate: `blocks` blocks of 256 threads, each thread
    32 x iters independent fp32 multiply-adds in registers (packed pairs or
    scalar fmaf); returns the (blocks,) output, every entry 496 + 32 * iters.
    Time it with events on `stream`: 2 * 32 * iters * 256 * blocks flops."""
    torch = _torch()
    if out is None:
        out = torch.empty(blocks, dtype=torch.float32, device="cuda")
    _check(lib().mpg_probe_fma_rate(out.data_ptr(), int(blocks), int(iters), 1 if packed else 0,
                                    _stream_handle(stream)))
    return out


def probe_tmem_acc_pair(A16, Bt16, stream=None):
    """One k-block (K = 64) of the CTA-pair tcgen05 path (M = 256) on fp16 A
    (256 x 64) and Bt (n x 64, row j = column j of B); returns the raw
    tcgen05.ld registers as a (2 CTAs, 4 warps, 32 lanes, n/32 loads, 32 regs)
    tensor."""
    torch = _torch()
    a = A16.to(torch.float16).contiguous()
    bt = Bt16.to(torch.float16).contiguous()
    n = bt.shape[0]
    if a.shape != (256, 64) or bt.shape[1] != 64:
        raise ValueError("A must be 256 x 64 and Bt n x 64")
    d = torch.empty((2, 4, 32, n // 32, 32), dtype=torch.float32, device=a.device)
    _check(lib().mpg_probe_tmem_acc_pair(a.data_ptr(), bt.data_ptr(), n, d.data_ptr(), _stream_handle(stream)))
    return d


def probe_epilogue_staging(blocks_in, scalar=False, stream=None):
    """Copy (nblocks, 32, 32) fp32 blocks through the epilogue's staging
    layout (mpg_probe_epilogue_staging); returns the copy."""
    torch = _torch()
    x = blocks_in.to(torch.float32).contiguous()
    if x.numel() % 1024 != 0:
        raise ValueError("blocks of 32 x 32 floats expected")
    out = torch.empty_like(x)
    _check(lib().mpg_probe_epilogue_staging(x.data_ptr(), out.data_ptr(), x.numel() // 1024, 1 if scalar else 0,
                                            _stream_handle(stream)))
    return out


def selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return lib().mpg_selftest_wait_timeout(timeout_ns, _stream_handle(stream))
