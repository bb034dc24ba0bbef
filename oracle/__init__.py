"""ORACLE — test infrastructure only.

A plain, slow, obviously-correct FP64 CPU reference for C = alpha*A*B + beta*C0
(see ``ref_gemm.c`` for the passages it follows and the readings it takes).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The GPU library
(``mixed_precision_matmul_gb300``) never imports it, and this package imports
nothing from the GPU library: the two share no code.

The C source is compiled with gcc into ``oracle/_build/liboracle.so`` by
:func:`build`; every function here is a thin ctypes call into that library plus
numpy plumbing.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_gemm.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# storage types
F32, F16, BF16, F64 = 0, 1, 2, 3
# operand quantisation
Q_NONE, Q_FP16, Q_BF16, Q_TF32_TRUNC, Q_TF32_RNA, Q_TF32_RNE, Q_SPLIT3, Q_SPLIT1, Q_SPLIT4 = range(9)

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, no fast-math); returns the .so path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, i32, dbl, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_void_p
        lib.orc_round_format.argtypes = [dbl, i32, i32, i32]
        lib.orc_round_format.restype = dbl
        for name in ("orc_fp16", "orc_bf16", "orc_tf32_rne", "orc_tf32_trunc", "orc_tf32_rna"):
            getattr(lib, name).argtypes = [dbl]
            getattr(lib, name).restype = dbl
        lib.orc_fp16_decode.argtypes = [ctypes.c_uint16]
        lib.orc_fp16_decode.restype = dbl
        lib.orc_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_decode.restype = dbl
        lib.orc_split.argtypes = [dbl, i32, i32, ctypes.POINTER(dbl), ctypes.POINTER(dbl)]
        lib.orc_split.restype = None
        lib.orc_quantize.argtypes = [vp, i32, i64, i64, i64, i32, i32, i32, vp, vp]
        lib.orc_quantize.restype = None
        lib.orc_gemm_f64.argtypes = [i64, i64, i64, vp, vp, vp, vp, i32, vp, i64, dbl, dbl,
                                     vp, vp, i64, i32]
        lib.orc_gemm_f64.restype = i32
        lib.orc_attention_f64.argtypes = [i64, i64, i64, i64, vp, vp, vp, dbl, vp, vp, i32]
        lib.orc_attention_f64.restype = i32
        lib.orc_gemm_points.argtypes = [i64,
                                        vp, i32, i64, i32, i32, i32,
                                        vp, i32, i64, i32, i32, i32,
                                        vp, i64, dbl, dbl, i64, vp, vp, vp, vp, i32]
        lib.orc_gemm_points.restype = i32
        lib.orc_gemm_fma_chain_f32.argtypes = [i64, i64, i64, vp, vp, vp, i64, ctypes.c_float, ctypes.c_float, vp]
        lib.orc_gemm_fma_chain_f32.restype = i32
        lib.orc_acc_coords.argtypes = [i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
        lib.orc_acc_coords.restype = i32
        for nm in ("orc_frag_a_coords", "orc_frag_b_coords"):
            getattr(lib, nm).argtypes = [i32, i32, ctypes.POINTER(i32), ctypes.POINTER(i32)]
            getattr(lib, nm).restype = i32
        _lib = lib
        return lib


# ---------------------------------------------------------------------------
# scalar and array quantisers
# ---------------------------------------------------------------------------

def round_format(x: float, p: int, emin: int, emax: int) -> float:
    return _load().orc_round_format(float(x), p, emin, emax)


def fp16(x: float) -> float:
    return _load().orc_fp16(float(x))


def bf16(x: float) -> float:
    return _load().orc_bf16(float(x))


def fp16_decode(code: int) -> float:
    return _load().orc_fp16_decode(int(code) & 0xFFFF)


def bf16_decode(code: int) -> float:
    return _load().orc_bf16_decode(int(code) & 0xFFFF)


def split(x: float, s: int = 0, L: int = 11) -> tuple[float, float]:
    hi, lo = ctypes.c_double(), ctypes.c_double()
    _load().orc_split(float(x), int(s), int(L), ctypes.byref(hi), ctypes.byref(lo))
    return hi.value, lo.value


def _storage(x: np.ndarray) -> tuple[np.ndarray, int]:
    """Map a numpy array to (contiguous array, oracle storage type).

    16-bit codes are passed as uint16 with an explicit kind: float16 arrays are
    F16; bfloat16 data arrives as a uint16 array wrapped by :class:`Bf16`.
    """
    if isinstance(x, Bf16):
        return np.ascontiguousarray(x.codes, dtype=np.uint16), BF16
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype == np.float16:
        return np.ascontiguousarray(x).view(np.uint16), F16
    if x.dtype == np.float64:
        return np.ascontiguousarray(x), F64
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


class Bf16:
    """A bf16 matrix given by its raw 16-bit codes (numpy has no bfloat16)."""

    def __init__(self, codes: np.ndarray):
        self.codes = np.asarray(codes, dtype=np.uint16)
        self.shape = self.codes.shape

    def to_f64(self) -> np.ndarray:
        return (self.codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def quantize(x, q: int = Q_NONE, s: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Element-wise quantisation of a 2-D operand (logical layout kept).

    Returns (hi, lo) binary64 arrays of x's shape; lo is all zero outside the
    split modes.  ``s`` is the split's power-of-two operand scale exponent.
    """
    arr, typ = _storage(x)
    rows, cols = arr.shape
    hi = np.empty((rows, cols), dtype=np.float64)
    lo = np.empty((rows, cols), dtype=np.float64)
    _load().orc_quantize(arr.ctypes.data, typ, rows, cols, cols, 0, q, s,
                         hi.ctypes.data, lo.ctypes.data)
    return hi, lo


# ---------------------------------------------------------------------------
# the product
# ---------------------------------------------------------------------------

def gemm(A, B, C0=None, alpha: float = 1.0, beta: float = 0.0,
         a_q: int = Q_NONE, b_q: int = Q_NONE, a_s: int = 0, b_s: int = 0,
         nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Full-grid reference.  A (m x k) and B (k x n) are logical matrices
    (numpy float32/float16/float64 or :class:`Bf16`).  Returns (ref, den):

    ref = alpha * sum_k q(A)[i,k] q(B)[k,j] + beta * C0[i,j]
    den = |alpha| * sum_k |q(A)[i,k]| |q(B)[k,j]| + |beta| |C0[i,j]|

    where for the split modes q(x) = hi + lo and the product keeps
    hi*hi + hi*lo + lo*hi (and lo*lo for Q_SPLIT4).
    """
    lib = _load()
    Ahi, Alo = quantize(A, a_q, a_s)
    Bhi, Blo = quantize(B, b_q, b_s)
    m, k = Ahi.shape
    k2, n = Bhi.shape
    if k != k2:
        raise ValueError("inner dimensions differ")
    split = 2 if a_q == Q_SPLIT4 else int(a_q in (Q_SPLIT3, Q_SPLIT1))
    ref = np.empty((m, n), dtype=np.float64)
    den = np.empty((m, n), dtype=np.float64)
    if C0 is not None:
        C0 = np.ascontiguousarray(C0, dtype=np.float32)
        c_ptr, ldc0 = C0.ctypes.data, C0.shape[1]
    else:
        c_ptr, ldc0 = None, n
    rc = lib.orc_gemm_f64(m, n, k, Ahi.ctypes.data, Alo.ctypes.data, Bhi.ctypes.data,
                          Blo.ctypes.data, split, c_ptr, ldc0, float(alpha), float(beta),
                          ref.ctypes.data, den.ctypes.data, n, nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the shape")
    return ref, den


def attention(Q, K, V, scale: float, q_q: int = Q_NONE, q_s: int = 0,
              nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Reference of the prompt-attention pair ("qsa_prompt_attn: ...",
    section "What's going on": scores q.k, row softmax, then p.v), in
    binary64.  Q is lq x d, K is lk x d and V is lk x dv (numpy
    float32/float16/float64 or :class:`Bf16`).  Q is first quantised by q_q (Q_SPLIT3: the value
    hi + lo of the split); K and V are taken as stored.  Returns (O, den):

    O[i, t]   = sum_j softmax_j(scale * q_i . k_j) V[j, t]
    den[i, t] = sum_j softmax_j(scale * q_i . k_j) |V[j, t]|
    """
    lib = _load()
    qh, ql = quantize(Q, q_q, q_s)
    qv = np.ascontiguousarray(qh + ql, dtype=np.float64)
    kv = _values(K)
    vv = _values(V)
    lq, d = qv.shape
    lk, dv = vv.shape
    if kv.shape != (lk, d):
        raise ValueError("attention operand shapes disagree")
    o = np.empty((lq, dv), dtype=np.float64)
    den = np.empty((lq, dv), dtype=np.float64)
    rc = lib.orc_attention_f64(lq, lk, d, dv, qv.ctypes.data, kv.ctypes.data, vv.ctypes.data, float(scale),
                               o.ctypes.data, den.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the attention shape")
    return o, den


def _values(X) -> np.ndarray:
    """Stored values of a matrix as a dense binary64 array (exact)."""
    if isinstance(X, Bf16):
        return np.ascontiguousarray(X.to_f64())
    return np.ascontiguousarray(np.asarray(X).astype(np.float64))


def gemm_points(A, B, k: int, rows, cols, C0=None, alpha: float = 1.0, beta: float = 0.0,
                a_q: int = Q_NONE, b_q: int = Q_NONE, a_s: int = 0, b_s: int = 0,
                a_col_major: bool = False, b_col_major: bool = False,
                lda: int | None = None, ldb: int | None = None,
                nthreads: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """Reference values of selected output elements (rows[p], cols[p]).

    A and B are given as STORED 2-D arrays: a row-major A is (m x lda) with
    the logical matrix in its first k columns; a column-major A is stored as
    (k x lda) holding A^T.  Same for B.  C0 (if given) is row-major 2-D.
    """
    lib = _load()
    a_arr, a_typ = _storage(A)
    b_arr, b_typ = _storage(B)
    lda = a_arr.shape[1] if lda is None else lda
    ldb = b_arr.shape[1] if ldb is None else ldb
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    npts = rows.shape[0]
    ref = np.empty(npts, dtype=np.float64)
    den = np.empty(npts, dtype=np.float64)
    if C0 is not None:
        c_ptr, ldc0 = C0.ctypes.data, C0.strides[0] // 4
        if C0.dtype != np.float32 or C0.strides[1] != 4:
            raise TypeError("C0 must be a row-major float32 array")
    else:
        c_ptr, ldc0 = None, 0
    rc = lib.orc_gemm_points(k, a_arr.ctypes.data, a_typ, lda, int(a_col_major), a_q, a_s,
                             b_arr.ctypes.data, b_typ, ldb, int(b_col_major), b_q, b_s,
                             c_ptr, ldc0, float(alpha), float(beta), npts,
                             rows.ctypes.data, cols.ctypes.data,
                             ref.ctypes.data, den.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return ref, den


def gemm_fma_chain_f32(A, B, C0=None, alpha: float = 1.0, beta: float = 0.0) -> np.ndarray:
    """The plain fp32 comparator's result, exactly: per element one fmaf
    chain over k ascending from +0, then alpha*acc (beta == 0, C0 unread)
    or fmaf(beta, C0, alpha*acc), all in fp32.  A (m x k), B (k x n), C0
    (m x n) are logical row-major values, cast to float32."""
    lib = _load()
    A = np.ascontiguousarray(A, dtype=np.float32)
    B = np.ascontiguousarray(B, dtype=np.float32)
    m, k = A.shape
    n = B.shape[1]
    if B.shape[0] != k:
        raise ValueError("inner dimensions differ")
    out = np.empty((m, n), dtype=np.float32)
    c_ptr, ldc0 = None, 0
    if C0 is not None:
        C0 = np.ascontiguousarray(C0, dtype=np.float32)
        c_ptr, ldc0 = C0.ctypes.data, n
    rc = lib.orc_gemm_fma_chain_f32(m, n, k, A.ctypes.data, B.ctypes.data, c_ptr, ldc0,
                                    float(np.float32(alpha)), float(np.float32(beta)), out.ctypes.data)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def max_rel_err(C: np.ndarray, ref: np.ndarray, den: np.ndarray) -> float:
    """max |C - ref| / den over all elements (the normalised error measure).

    Where den is 0 the numerator must be 0 as well (else the error is inf)."""
    C = np.asarray(C, dtype=np.float64)
    diff = np.abs(C - ref)
    zero = den == 0
    if np.any(diff[zero] != 0) or np.any(~np.isfinite(C)):
        return float("inf")
    if np.all(zero):
        return 0.0
    return float(np.max(diff[~zero] / den[~zero]))


def acc_coords(lane: int, j: int) -> tuple[int, int]:
    """(row, col) in the 16x8 tile of f32 accumulator value j of lane `lane`."""
    r, c = ctypes.c_int(), ctypes.c_int()
    if _load().orc_acc_coords(lane, j, ctypes.byref(r), ctypes.byref(c)) != 0:
        raise ValueError("lane or fragment index out of range")
    return r.value, c.value


def frag_a_coords(lane: int, i: int) -> tuple[int, int]:
    """(row, col) of value i of an m16n8k16 A fragment (PTX operand layout)."""
    r, c = ctypes.c_int(), ctypes.c_int()
    if _load().orc_frag_a_coords(lane, i, ctypes.byref(r), ctypes.byref(c)) != 0:
        raise ValueError("lane or value index out of range")
    return r.value, c.value


def frag_b_coords(lane: int, i: int) -> tuple[int, int]:
    """(k, n) of value i of an m16n8k16 B fragment (PTX operand layout)."""
    r, c = ctypes.c_int(), ctypes.c_int()
    if _load().orc_frag_b_coords(lane, i, ctypes.byref(r), ctypes.byref(c)) != 0:
        raise ValueError("lane or value index out of range")
    return r.value, c.value
