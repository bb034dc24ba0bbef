"""Pins of the oracle's attention (scores q.k, row softmax, p.v in binary64)
against closed forms, invariants and an independent library, so that a
dropped scale, a missing max subtraction, a softmax over the wrong axis or a
transposed V fails here."""
import math

import numpy as np
import pytest

import synthetic


def test_one_dominant_key_selects_its_value_row(orc):
    # key 1 scores 1000 above the others: exp(-1000) underflows to zero, so
    # the weights are exactly one-hot.  Without the max subtraction exp(1000)
    # overflows; reading V transposed picks a column instead of row 1.
    d = 6
    Q = np.zeros((2, d), np.float32)
    Q[:, 0] = 1.0
    K = np.zeros((3, d), np.float32)
    K[1, 0] = 1000.0
    V = synthetic.asymmetric((3, d), 201)
    O, den = orc.attention(Q, K, V, scale=1.0)
    assert np.array_equal(O, np.repeat(V[1:2].astype(np.float64), 2, axis=0))
    assert np.array_equal(den, np.abs(O))


def test_identical_keys_and_zero_query_give_the_mean_of_v(orc):
    V = synthetic.normal((37, 5), 202)
    mean = V.astype(np.float64).mean(axis=0)
    K = np.repeat(synthetic.normal((1, 5), 203), 37, axis=0)
    Q = synthetic.normal((3, 5), 204)
    O, _ = orc.attention(Q, K, V, scale=0.7)
    assert np.max(np.abs(O - mean)) < 1e-15
    O, _ = orc.attention(np.zeros((2, 5), np.float32), synthetic.normal((37, 5), 205), V, scale=1.3)
    assert np.max(np.abs(O - mean)) < 1e-15


def test_two_keys_reduce_to_the_logistic_function(orc):
    # two keys: p_0 = 1 / (1 + exp(-(s_0 - s_1))) with s_j = scale * q . k_j;
    # several different queries (rows) and a scale that is not 1
    g = np.random.Generator(np.random.PCG64(206))
    d, scale = 4, 0.375
    Q = g.integers(-3, 4, size=(5, d)).astype(np.float32)
    K = g.integers(-3, 4, size=(2, d)).astype(np.float32)
    V = g.integers(-9, 10, size=(2, 3)).astype(np.float32)
    O, _ = orc.attention(Q, K, V, scale=scale)
    for i in range(5):
        s0 = scale * sum(float(Q[i, t]) * float(K[0, t]) for t in range(d))
        s1 = scale * sum(float(Q[i, t]) * float(K[1, t]) for t in range(d))
        p0 = 1.0 / (1.0 + math.exp(-(s0 - s1)))
        expect = p0 * V[0].astype(np.float64) + (1.0 - p0) * V[1].astype(np.float64)
        assert np.max(np.abs(O[i] - expect)) < 1e-14


def test_key_order_does_not_matter(orc):
    Q = synthetic.normal((4, 16), 207)
    K = synthetic.normal((50, 16), 208)
    V = synthetic.normal((50, 8), 209)
    O, den = orc.attention(Q, K, V, scale=0.25)
    perm = np.random.Generator(np.random.PCG64(210)).permutation(50)
    Op, denp = orc.attention(Q, K[perm], V[perm], scale=0.25)
    assert np.max(np.abs(O - Op)) < 1e-14 and np.max(np.abs(den - denp)) < 1e-14


def test_nonnegative_values_make_den_equal_o(orc):
    Q = synthetic.normal((3, 8), 211)
    K = synthetic.normal((20, 8), 212)
    V = np.abs(synthetic.normal((20, 4), 213))
    O, den = orc.attention(Q, K, V, scale=0.5)
    assert np.array_equal(O, den)


def test_against_scipy_softmax(orc):
    special = pytest.importorskip("scipy.special")
    Q = synthetic.normal((9, 32), 214)
    K = synthetic.normal((70, 32), 215).astype(np.float16)
    V = synthetic.normal((70, 12), 216).astype(np.float16)
    scale = 2.0 / math.sqrt(32)
    O, den = orc.attention(Q, K, V, scale=scale)
    S = scale * (Q.astype(np.float64) @ K.astype(np.float64).T)
    P = special.softmax(S, axis=1)
    assert np.max(np.abs(O - P @ V.astype(np.float64))) < 1e-13
    assert np.max(np.abs(den - P @ np.abs(V.astype(np.float64)))) < 1e-13


def test_split_query_is_the_hi_plus_lo_value(orc):
    # mode Q of the attention: q replaced by the value of its split, which
    # differs from q by at most a few units of 2^-22 relative
    Q = synthetic.normal((6, 16), 217)
    K = synthetic.normal((30, 16), 218).astype(np.float16)
    V = synthetic.normal((30, 16), 219).astype(np.float16)
    OR, _ = orc.attention(Q, K, V, scale=0.3)
    OQ, den = orc.attention(Q, K, V, scale=0.3, q_q=orc.Q_SPLIT3)
    hi, lo = orc.quantize(Q, orc.Q_SPLIT3)
    q = Q.astype(np.float64)
    assert np.max(np.abs(hi + lo - q) / np.abs(q)) <= 2.0 ** -21
    assert 0 < np.max(np.abs(OR - OQ) / den) < 1e-6


def test_zero_scale_gives_the_mean_of_v(orc):
    # scale 0: every score is 0 whatever q and k, the weights uniform.  A
    # scale applied to V or to the output instead of the scores fails here.
    Q = synthetic.normal((4, 7), 206)
    K = synthetic.normal((29, 7), 207)
    V = synthetic.normal((29, 7), 208)
    O, _ = orc.attention(Q, K, V, scale=0.0)
    assert np.max(np.abs(O - V.astype(np.float64).mean(axis=0))) < 1e-15


def test_a_common_shift_of_the_keys_leaves_o_unchanged(orc):
    # k_j -> k_j + u adds scale * q_i . u to every score of row i: the
    # softmax of a row does not change (binary64 inputs, so the shift is
    # exact in the scores up to rounding).  A softmax over the query axis
    # changes O here: the shifts differ from row to row.
    Q = synthetic.normal((5, 8), 209).astype(np.float64)
    K = synthetic.normal((41, 8), 210).astype(np.float64)
    V = synthetic.normal((41, 8), 211).astype(np.float64)
    u = 3.0 * synthetic.normal((1, 8), 212).astype(np.float64)
    O1, _ = orc.attention(Q, K, V, scale=0.6)
    O2, _ = orc.attention(Q, K + u, V, scale=0.6)
    assert np.max(np.abs(O1 - O2)) < 1e-12
    # and the per-row shifts differ (so a softmax over the wrong axis would show)
    assert np.ptp(Q @ u.T) > 1.0
