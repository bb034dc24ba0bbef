"""Pins of the oracle's product against brute force, closed forms and an
independent library (numpy float64 matmul), so that a dropped term, a wrong
sign or index, or a transposed operand in the oracle fails here."""
import numpy as np
import pytest

import synthetic


def test_brute_force_16x8x16_small_integers(orc):
    g = np.random.Generator(np.random.PCG64(21))
    A = g.integers(-8, 9, size=(16, 16))
    B = g.integers(-8, 9, size=(16, 8))
    C0 = g.integers(-8, 9, size=(16, 8))
    ref, den = orc.gemm(A.astype(np.float32), B.astype(np.float32), C0.astype(np.float32),
                        alpha=3.0, beta=-2.0)
    for i in range(16):
        for j in range(8):
            s = sum(int(A[i, k]) * int(B[k, j]) for k in range(16))
            d = sum(abs(int(A[i, k])) * abs(int(B[k, j])) for k in range(16))
            assert ref[i, j] == 3 * s - 2 * int(C0[i, j])
            assert den[i, j] == 3 * d + 2 * abs(int(C0[i, j]))


def test_identity_and_permutation_exact(orc):
    A = synthetic.asymmetric((24, 24), 22)
    I = np.eye(24, dtype=np.float32)
    ref, _ = orc.gemm(A, I)
    assert np.array_equal(ref, A.astype(np.float64))
    ref, _ = orc.gemm(I, A)
    assert np.array_equal(ref, A.astype(np.float64))
    perm = np.random.Generator(np.random.PCG64(23)).permutation(24)
    P = np.eye(24, dtype=np.float32)[perm]
    ref, _ = orc.gemm(P, A)
    assert np.array_equal(ref, A[perm].astype(np.float64))
    ref, _ = orc.gemm(A, P.T.copy())
    assert np.array_equal(ref, A[:, perm].astype(np.float64))


def test_rank1_closed_form(orc):
    g = np.random.Generator(np.random.PCG64(24))
    u, v, w, z = (g.integers(-50, 51, size=n).astype(np.float32) for n in (12, 20, 20, 9))
    A = np.outer(u, v).astype(np.float32)
    B = np.outer(w, z).astype(np.float32)
    ref, _ = orc.gemm(A, B)
    vw = float(np.dot(v.astype(np.float64), w.astype(np.float64)))
    assert np.array_equal(ref, vw * np.outer(u.astype(np.float64), z.astype(np.float64)))


def test_alpha_beta_and_empty_k(orc):
    A = synthetic.uniform((5, 0), 1)
    B = synthetic.uniform((0, 7), 2)
    C0 = synthetic.uniform((5, 7), 3)
    ref, den = orc.gemm(A, B, C0, alpha=2.0, beta=0.25)
    assert np.array_equal(ref, 0.25 * C0.astype(np.float64))
    assert np.array_equal(den, 0.25 * np.abs(C0.astype(np.float64)))
    A = synthetic.uniform((5, 6), 1)
    B = synthetic.uniform((6, 7), 2)
    ref, _ = orc.gemm(A, B, C0, alpha=0.0, beta=1.0)
    assert np.array_equal(ref, C0.astype(np.float64))


def test_against_numpy_float64_matmul(orc):
    A = synthetic.uniform((37, 53), 1)
    B = synthetic.uniform((53, 29), 2)
    C0 = synthetic.uniform((37, 29), 3)
    ref, den = orc.gemm(A, B, C0, alpha=1.5, beta=-0.75)
    Ad, Bd, Cd = (x.astype(np.float64) for x in (A, B, C0))
    exp = 1.5 * (Ad @ Bd) - 0.75 * Cd
    expd = 1.5 * (np.abs(Ad) @ np.abs(Bd)) + 0.75 * np.abs(Cd)
    assert np.max(np.abs(ref - exp) / expd) < 1e-14
    assert np.max(np.abs(den - expd) / expd) < 1e-14


def test_quantised_modes_against_numpy_conversions(orc):
    A = synthetic.uniform((19, 40), 1)
    B = synthetic.uniform((40, 23), 2)
    ref, _ = orc.gemm(A, B, a_q=orc.Q_FP16, b_q=orc.Q_FP16)
    Ah = A.astype(np.float16).astype(np.float64)
    Bh = B.astype(np.float16).astype(np.float64)
    assert np.max(np.abs(ref - Ah @ Bh)) < 1e-13


def test_split_drops_exactly_the_lo_lo_term(orc):
    # inputs that split exactly into hi + lo: fp16 value plus a small fp16
    # multiple of 2^-12, so mode R and the three-chain sum differ by sum lo*lo
    g = np.random.Generator(np.random.PCG64(25))
    def exact_split(shape):
        hi = g.integers(1024, 2048, size=shape) / 1024.0 * np.where(g.integers(0, 2, shape) == 0, -1, 1)
        lo = g.integers(-255, 256, size=shape) * 2.0 ** -20
        return (hi + lo).astype(np.float32), hi, lo
    A, Ah, Al = exact_split((9, 31))
    B, Bh, Bl = exact_split((31, 11))
    rR, _ = orc.gemm(A, B)
    rQ, _ = orc.gemm(A, B, a_q=orc.Q_SPLIT3, b_q=orc.Q_SPLIT3)
    assert np.max(np.abs((rR - rQ) - Al @ Bl)) < 1e-18
    assert np.max(np.abs(rQ - (Ah @ Bh + Ah @ Bl + Al @ Bh))) < 1e-13


def test_points_match_full_grid_for_every_layout(orc):
    m, n, k = 21, 17, 33
    A = synthetic.asymmetric((m, k), 31)
    B = synthetic.asymmetric((k, n), 32)
    C0 = synthetic.uniform((m, n), 3)
    full, fden = orc.gemm(A, B, C0, 1.25, 0.5, orc.Q_FP16, orc.Q_FP16)
    rows, cols = np.meshgrid(np.arange(m), np.arange(n), indexing="ij")
    rows, cols = rows.ravel(), cols.ravel()
    for a_cm in (False, True):
        for b_cm in (False, True):
            a_st = synthetic.padded(k, m, m + 3, A.T) if a_cm else synthetic.padded(m, k, k + 5, A)
            b_st = synthetic.padded(n, k, k + 2, B.T) if b_cm else synthetic.padded(k, n, n + 7, B)
            ref, den = orc.gemm_points(a_st, b_st, k, rows, cols, C0, 1.25, 0.5,
                                       orc.Q_FP16, orc.Q_FP16,
                                       a_col_major=a_cm, b_col_major=b_cm)
            assert np.array_equal(ref, full.ravel())
            assert np.array_equal(den, fden.ravel())


def test_transposed_operand_is_detected(orc):
    # a plausible layout mistake (reading A as its transpose) must change the
    # result on asymmetric, non-repeating inputs
    A = synthetic.asymmetric((16, 16), 41)
    B = synthetic.asymmetric((16, 8), 42)
    ref, _ = orc.gemm(A, B)
    wrong, _ = orc.gemm(A.T.copy(), B)
    assert np.count_nonzero(ref != wrong) == ref.size


def test_bf16_storage_is_read_exactly(orc):
    x = synthetic.normal((8, 12), 1)
    codes = synthetic.bf16_codes_from_f32(x)
    b = orc.Bf16(codes)
    vals = b.to_f64()
    I = np.eye(12, dtype=np.float32)
    ref, _ = orc.gemm(b, I)
    assert np.array_equal(ref, vals)


def test_max_rel_err(orc):
    ref = np.array([1.0, -2.0, 0.0])
    den = np.array([2.0, 4.0, 0.0])
    assert orc.max_rel_err(np.array([1.5, -2.0, 0.0]), ref, den) == 0.25
    assert orc.max_rel_err(np.array([1.0, -2.0, 1e-30]), ref, den) == float("inf")
    assert orc.max_rel_err(np.array([np.nan, -2.0, 0.0]), ref, den) == float("inf")


def test_split_of_a_only_with_fp16_b(orc):
    # A splits exactly into hi + lo (fp16 value plus a small multiple of
    # 2^-20) and B holds fp16 values: the problem on the quantised inputs of
    # the A-only split (A = hi + lo, B = fp16(B)) is then the exact product
    g = np.random.Generator(np.random.PCG64(26))
    hi = g.integers(1024, 2048, size=(7, 29)) / 1024.0
    lo = g.integers(-255, 256, size=(7, 29)) * 2.0 ** -20
    A = (hi + lo).astype(np.float32)
    B = (g.integers(-2048, 2049, size=(29, 13)) / 256.0).astype(np.float32)   # exact in fp16
    rR, _ = orc.gemm(A, B)
    rQ, _ = orc.gemm(A, B, a_q=orc.Q_SPLIT3, b_q=orc.Q_FP16)
    assert np.array_equal(rR, rQ)
    # B values that are not fp16 numbers are rounded: the difference is A times
    # the rounding error of B, which numpy's float16 conversion supplies
    B2 = synthetic.uniform((29, 13), 27)
    rR2, _ = orc.gemm(A, B2)
    rQ2, _ = orc.gemm(A, B2, a_q=orc.Q_SPLIT3, b_q=orc.Q_FP16)
    expect = A.astype(np.float64) @ (B2.astype(np.float16).astype(np.float64) - B2.astype(np.float64))
    assert np.max(np.abs((rQ2 - rR2) - expect)) < 1e-12


def test_four_chain_split_keeps_lo_lo(orc):
    # inputs that split exactly into hi + lo: with lo*lo kept the four-term
    # sum is the exact product; the three-term sum misses exactly sum lo*lo
    g = np.random.Generator(np.random.PCG64(28))
    def exact_split(shape):
        hi = g.integers(1024, 2048, size=shape) / 1024.0 * np.where(g.integers(0, 2, shape) == 0, -1, 1)
        lo = g.integers(-255, 256, size=shape) * 2.0 ** -20
        return (hi + lo).astype(np.float32), lo
    A, Al = exact_split((8, 27))
    B, Bl = exact_split((27, 10))
    rR, _ = orc.gemm(A, B)
    r4, _ = orc.gemm(A, B, a_q=orc.Q_SPLIT4, b_q=orc.Q_SPLIT4)
    r3, _ = orc.gemm(A, B, a_q=orc.Q_SPLIT3, b_q=orc.Q_SPLIT3)
    assert np.array_equal(r4, rR)
    assert np.max(np.abs((r4 - r3) - Al @ Bl)) < 1e-18
    rows, cols = np.array([0, 3, 7]), np.array([9, 0, 4])
    p4, _ = orc.gemm_points(A, B, 27, rows, cols, a_q=orc.Q_SPLIT4, b_q=orc.Q_SPLIT4)
    assert np.array_equal(p4, rR[rows, cols])


# ---- the fp32 comparator's exact result (one fmaf chain per element)

def test_fma_chain_is_fused_and_ascending(orc):
    """k = 2: -1 * 1, then (1 + 2^-12)^2 - 1 in ONE rounding gives
    2^-11 + 2^-24 exactly; a separate multiply would round the square to
    1 + 2^-11 first (a tie to even) and give 2^-11, and the descending
    order (square first) gives 2^-11 too."""
    x = 1.0 + 2.0 ** -12
    out = orc.gemm_fma_chain_f32(np.array([[-1.0, x]]), np.array([[1.0], [x]]))
    assert out[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)


def test_fma_chain_order_decides_cancellation(orc):
    """1 + 2^24 - 2^24 in k order: 1 + 2^24 rounds to 2^24 (a tie to even),
    so the chain ends at 0 although the exact sum is 1."""
    out = orc.gemm_fma_chain_f32(np.array([[1.0, 2.0 ** 24, -(2.0 ** 24)]]), np.ones((3, 1)))
    assert out[0, 0] == 0.0
    out = orc.gemm_fma_chain_f32(np.array([[-(2.0 ** 24), 2.0 ** 24, 1.0]]), np.ones((3, 1)))
    assert out[0, 0] == 1.0


def test_fma_chain_small_integers_exact(orc):
    g = np.random.Generator(np.random.PCG64(31))
    A = g.integers(-8, 9, size=(9, 40))
    B = g.integers(-8, 9, size=(40, 7))
    out = orc.gemm_fma_chain_f32(A, B)
    assert np.array_equal(out.astype(np.int64), A @ B)


def test_fma_chain_epilogue_roundings(orc):
    """alpha * acc is rounded to fp32 on its own, then beta * C0 is added in
    one fmaf: acc = 3, alpha = 1 + 2^-23 gives t = 3 + 2^-21 (1.5 ulp, a tie
    to even), and fmaf(1, -3, t) = 2^-21.  Fusing alpha instead would give
    3 * 2^-23.  With beta = 0 C0 is not read (NaN stays out)."""
    one = np.ones((1, 1))
    out = orc.gemm_fma_chain_f32(np.array([[3.0]]), one, np.array([[-3.0]]), alpha=1.0 + 2.0 ** -23, beta=1.0)
    assert out[0, 0] == np.float32(2.0 ** -21)
    x = 1.0 + 2.0 ** -12
    out = orc.gemm_fma_chain_f32(np.array([[-1.0]]), one, np.array([[x]]), alpha=1.0, beta=x)
    assert out[0, 0] == np.float32(2.0 ** -11 + 2.0 ** -24)
    out = orc.gemm_fma_chain_f32(np.array([[2.0]]), one, np.array([[np.nan]]), alpha=0.5, beta=0.0)
    assert out[0, 0] == 1.0
    assert orc.gemm_fma_chain_f32(np.zeros((2, 0)), np.zeros((0, 3)), np.full((2, 3), 4.0), 1.0, 0.5).tolist() == \
        [[2.0] * 3] * 2


def test_fma_chain_within_the_recursive_summation_bound(orc):
    """|chain - exact| <= gamma_k * sum |a||b| with gamma_k = k u / (1 - k u),
    u = 2^-24 (the error bound of recursive summation with fused steps),
    the exact value from the fp64 reference on the same fp32 inputs."""
    g = np.random.Generator(np.random.PCG64(32))
    m, n, k = 20, 17, 300
    A = g.standard_normal((m, k)).astype(np.float32)
    B = g.standard_normal((k, n)).astype(np.float32)
    out = orc.gemm_fma_chain_f32(A, B)
    ref, den = orc.gemm(A, B)
    u = 2.0 ** -24
    gamma = k * u / (1 - k * u)
    err = np.abs(out.astype(np.float64) - ref)
    assert np.all(err <= gamma * den)
    assert np.max(err / den) > 0          # and it is not the fp64 value
