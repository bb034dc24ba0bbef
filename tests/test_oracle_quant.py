"""Pins of the oracle's quantisers against things other than the oracle:
numpy's float16 conversion, PyTorch's bfloat16 conversion, IEEE special values
and the algebraic invariants of the hi/lo split."""
import math

import numpy as np
import pytest
import torch

import synthetic


def _q(orc, x, q, s=0):
    hi, lo = orc.quantize(np.asarray(x, dtype=np.float64).reshape(1, -1), q, s)
    return hi.ravel(), lo.ravel()


def test_fp16_decode_all_codes_matches_numpy(orc):
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    mine = np.array([orc.fp16_decode(int(c)) for c in codes])
    fin = np.isfinite(ref)
    assert np.array_equal(mine[fin], ref[fin])
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    assert np.array_equal(mine[np.isinf(ref)], ref[np.isinf(ref)])


def test_fp16_round_trip_every_finite_code(orc):
    vals = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float64)
    vals = vals[np.isfinite(vals)]
    hi, _ = _q(orc, vals, orc.Q_FP16)
    assert np.array_equal(hi, vals)


def test_fp16_matches_numpy_on_random_fp32(orc):
    g = np.random.Generator(np.random.PCG64(11))
    # wide exponent range: subnormals, normals and overflow
    x = (g.standard_normal(400_000) * np.exp2(g.uniform(-30, 18, 400_000))).astype(np.float32)
    hi, _ = _q(orc, x.astype(np.float64), orc.Q_FP16)
    ref = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(hi, ref)


@pytest.mark.parametrize("x,expect", [
    (1.0 + 2.0 ** -11, 1.0),                       # tie -> even (down)
    (1.0 + 3 * 2.0 ** -11, 1.0 + 2.0 ** -9),       # tie -> even (up)
    (65519.99, 65504.0),                           # just below the overflow midpoint
    (65520.0, math.inf),                           # overflow midpoint rounds to inf
    (2.0 ** -25, 0.0),                             # half the smallest subnormal -> 0 (even)
    (3 * 2.0 ** -25, 2.0 ** -23),                  # subnormal tie -> even
    (-(2.0 ** -14) * (1 - 2.0 ** -12), -(2.0 ** -14)),  # rounds up into the normal range
])
def test_fp16_special_cases(orc, x, expect):
    assert orc.fp16(x) == expect


def test_bf16_round_trip_and_torch_agreement(orc):
    codes = np.arange(65536, dtype=np.uint16)
    vals = (codes.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    fin = np.isfinite(vals)
    hi, _ = _q(orc, vals[fin], orc.Q_BF16)
    assert np.array_equal(hi, vals[fin])
    g = np.random.Generator(np.random.PCG64(12))
    x = (g.standard_normal(400_000) * np.exp2(g.uniform(-140, 127, 400_000))).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    hi, _ = _q(orc, x.astype(np.float64), orc.Q_BF16)
    assert np.array_equal(hi, ref)


def test_bf16_input_generator_is_exact_in_bf16(orc):
    codes = synthetic.bf16_codes_from_f32(synthetic.normal((64, 64), 1))
    vals = orc.Bf16(codes).to_f64().ravel()
    hi, _ = _q(orc, vals, orc.Q_BF16)
    assert np.array_equal(hi, vals)


def test_tf32_rne_equals_fp16_rounding_inside_fp16_range(orc):
    # tf32 and fp16 share the 11-bit significand, so where both are normal
    # their round-to-nearest-even results coincide; numpy supplies fp16.
    g = np.random.Generator(np.random.PCG64(13))
    x = (g.uniform(1.0, 2.0, 200_000) * np.exp2(g.integers(-14, 15, 200_000))).astype(np.float32)
    x *= np.where(g.integers(0, 2, x.size) == 0, -1, 1).astype(np.float32)
    hi, _ = _q(orc, x.astype(np.float64), orc.Q_TF32_RNE)
    ref = x.astype(np.float16).astype(np.float64)
    keep = np.isfinite(ref)
    assert np.array_equal(hi[keep], ref[keep])


def test_tf32_truncation_and_rna_properties(orc):
    g = np.random.Generator(np.random.PCG64(14))
    x = (g.standard_normal(100_000) * np.exp2(g.uniform(-100, 100, 100_000))).astype(np.float32)
    xd = x.astype(np.float64)
    tr, _ = _q(orc, xd, orc.Q_TF32_TRUNC)
    rna, _ = _q(orc, xd, orc.Q_TF32_RNA)
    rne, _ = _q(orc, xd, orc.Q_TF32_RNE)
    bits = tr.astype(np.float32).view(np.uint32)
    assert np.all(bits & 0x1FFF == 0)                # 10 fraction bits kept
    assert np.all(np.abs(tr) <= np.abs(xd))          # toward zero
    e = np.floor(np.log2(np.abs(xd)))
    ulp = np.exp2(e - 10)
    assert np.all(np.abs(xd - tr) < ulp)
    assert np.all(np.abs(xd - rna) <= ulp / 2)       # nearest
    assert np.all(np.abs(xd - rne) <= ulp / 2)
    # exact ties: rna goes away from zero, rne to the even neighbour
    t = np.float32(1.0 + 2.0 ** -11)
    assert orc.quantize(np.array([[t]], np.float64), orc.Q_TF32_RNA)[0][0, 0] == 1.0 + 2.0 ** -10
    assert orc.quantize(np.array([[t]], np.float64), orc.Q_TF32_RNE)[0][0, 0] == 1.0


def test_split_invariants(orc):
    g = np.random.Generator(np.random.PCG64(15))
    x = synthetic.loguniform_signed(50_000, 16).astype(np.float64)
    for q, L in ((orc.Q_SPLIT3, 11), (orc.Q_SPLIT1, 0)):
        hi, lo = _q(orc, x, q)
        # hi is x rounded to fp16 (numpy conversion)
        assert np.array_equal(hi, x.astype(np.float16).astype(np.float64))
        # the residual x - hi is exact in fp32
        r = x - hi
        assert np.array_equal(r.astype(np.float32).astype(np.float64), r)
        # lo is the residual rounded to fp16 after the 2^L scaling
        assert np.array_equal(lo * 2.0 ** L, (r * 2.0 ** L).astype(np.float16).astype(np.float64))
        # |lo| <= ulp(hi)/2
        e = np.floor(np.log2(np.abs(hi)))
        assert np.all(np.abs(lo) <= np.exp2(e - 11) * (1 + 1e-12))
    # with the 2^11 lo scale and inputs in [2^-8, 2^8] the pair carries ~22 bits
    hi, lo = _q(orc, x, orc.Q_SPLIT3)
    rel = np.abs(x - hi - lo) / np.abs(x)
    assert rel.max() <= 2.0 ** -21
    # without the scale, lo of |x| < 2^-3 falls into the fp16 subnormals
    hi1, lo1 = _q(orc, x, orc.Q_SPLIT1)
    rel1 = np.abs(x - hi1 - lo1) / np.abs(x)
    assert rel1.max() > rel.max()


def test_split_operand_scale_rescues_small_values(orc):
    # values far below 2^-14 sit in the fp16 subnormals even with the 2^11 lo
    # scale; a power-of-two operand scale keeps ~22 bits and is exactly undone
    x = np.array([3.7e-6, 1.0e-7, 4.1e-5, 0.012, 1e-9, 2e-8], dtype=np.float32).astype(np.float64)
    hi0, lo0 = _q(orc, x, orc.Q_SPLIT3, 0)
    hi, lo = _q(orc, x, orc.Q_SPLIT3, 14)
    assert np.max(np.abs(x - hi - lo) / x) <= 2.0 ** -21
    assert np.max(np.abs(x - hi0 - lo0) / x) > 2.0 ** -12
