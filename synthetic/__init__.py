"""Seeded synthetic inputs for the GEMM workloads.

This module only draws random numbers with numpy's PCG64 generator and lays
them out in memory (leading dimensions, padding, batch strides).  It holds none
of the product's arithmetic and no precision conversion of the method: it is
the one module that both the GPU tests/benchmark and the CPU oracle read their
inputs from, so that the two sides see the same bytes.

Workloads (shapes and distributions follow the pages' workloads; the recipes
are listed in the design notes):

* ``square_uniform``   256^3, fp32 U(-1,1), row-major, ld = 256.
* ``batched``          2048 x (64x64 = 64x4096 * 4096x64), fp32 U(-1,1),
                       A row-major, B column-major, lda = ldb = 4096 + 8,
                       C row-major with ldc = 64 + 8, packed batch strides.
* ``large_bf16``       8192^3, bf16 N(0,1) (fp32 normal draws stored as bf16),
                       C0 fp32 N(0,1), alpha = 1, beta = 0.5; and the tail
                       shape 8191 x 8177 x 8183 with unpadded leading dims.
* ``loguniform``       4096^3 fp32 with |x| = 2^u, u ~ U(-8, 8), random sign.
* ``attention``        Q 2048x128 and K 32768x128 ~ N(0,1)/sqrt(128);
                       P = row-softmax of N(0, 2^2) logits (2048 x 32768),
                       V 32768x128 ~ N(0,1).

Seeds: A = 1, B = 2, C0 = 3, Q = 4, K = 5, V = 6, logits = 7 (plus an offset
for callers that need several independent draws).
"""
from __future__ import annotations

import numpy as np

SEED_A, SEED_B, SEED_C0, SEED_Q, SEED_K, SEED_V, SEED_LOGITS = 1, 2, 3, 4, 5, 6, 7


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform(shape, seed: int, lo: float = -1.0, hi: float = 1.0) -> np.ndarray:
    return rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def normal(shape, seed: int, scale: float = 1.0) -> np.ndarray:
    return (rng(seed).standard_normal(size=shape, dtype=np.float32) * np.float32(scale))


def loguniform_signed(shape, seed: int, emin: float = -8.0, emax: float = 8.0) -> np.ndarray:
    """|x| = 2^u with u ~ U(emin, emax); the sign is +-1 with equal odds."""
    g = rng(seed)
    u = g.uniform(emin, emax, size=shape)
    sign = np.where(g.integers(0, 2, size=shape) == 0, -1.0, 1.0)
    return (sign * np.exp2(u)).astype(np.float32)


def bf16_codes_from_f32(x: np.ndarray) -> np.ndarray:
    """Store fp32 draws as bf16 (the storage format of the bf16 workloads).

    Uses PyTorch's CPU conversion (round to nearest even); the result is the
    raw 16-bit codes as uint16.
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def asymmetric(shape, seed: int) -> np.ndarray:
    """Distinct, non-repeating small values that expose a transposed or a
    half-swapped layout: a random permutation of 1..N scaled into (0, 1],
    with alternating signs by draw order.  Every value is exact in fp16."""
    n = int(np.prod(shape))
    perm = rng(seed).permutation(n) + 1
    vals = perm.astype(np.float64) / 2.0 ** np.ceil(np.log2(n + 1))
    vals = vals * np.where(np.arange(n) % 2 == 0, 1.0, -1.0)
    return vals.reshape(shape).astype(np.float32)


def padded(rows: int, cols: int, ld: int, fill: np.ndarray | None = None,
           dtype=np.float32, pad_value=0) -> np.ndarray:
    """A (rows x ld) buffer whose first `cols` columns hold `fill`."""
    buf = np.full((rows, ld), pad_value, dtype=dtype)
    if fill is not None:
        buf[:, :cols] = fill
    return buf


def softmax_rows_f64(logits: np.ndarray) -> np.ndarray:
    """Row softmax computed in binary64 (input preparation for the attention
    workload: P is defined as the softmax of the drawn logits)."""
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    np.exp(z, out=z)
    z /= z.sum(axis=1, keepdims=True)
    return z


def attention_fused_inputs(lq: int = 2048, lk: int = 32768, d: int = 128):
    """Operands of the fused prompt attention: Q fp32 N(0,1); K and V drawn
    N(0,1) and stored as fp16 (the key/value cache's storage type); the
    softmax scale 2/sqrt(d) gives the logits scale * q.k a standard
    deviation of 2, the spread of the attention workload's logits."""
    q = normal((lq, d), SEED_Q)
    k = normal((lk, d), SEED_K).astype(np.float16)
    v = normal((lk, d), SEED_V).astype(np.float16)
    return q, k, v, 2.0 / float(np.sqrt(d))


def attention_inputs(lq: int = 2048, lk: int = 32768, d: int = 128):
    q = normal((lq, d), SEED_Q, 1.0 / np.sqrt(d))
    k = normal((lk, d), SEED_K, 1.0 / np.sqrt(d))
    logits = normal((lq, lk), SEED_LOGITS, 2.0)
    p = softmax_rows_f64(logits).astype(np.float32)
    v = normal((lk, d), SEED_V, 1.0)
    return q, k, p, v
