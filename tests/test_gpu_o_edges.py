"""GPU: the converters on the values where conversion itself decides the
result ("Tensor Core operands: a matrix instruction still needs a layout
contract", fourth paragraph: overflow, underflow and output conversion stay
relevant; fifth: test difficult inputs).

Each output element is one product q(x) * b with every other product zero,
so the element shows what the conversion made of x: fp32 inputs at and
beyond fp16's overflow midpoint (65520 rounds to infinity), fp16 subnormals
(2^-15 .. 2^-24) including ties, bf16's overflow midpoint and subnormals,
and, for the split, values beyond its range (|x * 2^s| >= 65520 gives an
infinite hi and the documented non-finite result) and values whose lo half
lies in fp16's subnormals.  The GPU result is compared element by element
with the oracle on the quantised-input problem, inf against inf and NaN
against NaN, on the three paths that convert: in the load stage (TMA
staging), in the separate conversion pass, and with generic loads."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
from helpers import TOL, Case

pytestmark = pytest.mark.gpu

F16_MAX = 65504.0
FP16_SPECIALS = [
    F16_MAX, 65519.99, 65520.0, 65536.0, 1.0e6, np.inf, -65520.0, -65519.99, np.nan,
    2.0 ** -14, 2.0 ** -15, 2.0 ** -24, 2.0 ** -25, 1.5 * 2.0 ** -25, 2.0 ** -26, 3 * 2.0 ** -25,
    5 * 2.0 ** -25, 7 * 2.0 ** -25, float.fromhex("0x1.23456p-17"), float.fromhex("0x1.fffffep-15"),
    -(2.0 ** -24), -3 * 2.0 ** -25, 1.0, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 0.0, -0.0,
]
BF16_MAX = float.fromhex("0x1.fep127")
# near bf16's overflow midpoint (partners of magnitude <= 1 keep the finite
# products within fp32's range: bf16's largest value is just below fp32's)
BF16_LARGE = [
    BF16_MAX, float.fromhex("0x1.fefffep127"), float.fromhex("0x1.ffp127"), float.fromhex("0x1.fffffep127"),
    np.inf, -np.inf, -float.fromhex("0x1.ffp127"), np.nan, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 0.0,
]
# bf16 subnormals (2^-127 .. 2^-133) and ties; partners of 2^24 keep the
# products in fp32's normal range
BF16_SMALL = [
    2.0 ** -126, 2.0 ** -127, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 3 * 2.0 ** -134,
    float.fromhex("0x1.234p-130"), -(2.0 ** -133), float.fromhex("0x1.ff8p-127"), 1.0,
]
# split: hi overflows at |x * 2^s| >= 65520; lo of tiny values is subnormal
SPLIT_SPECIALS = [
    65519.99, 65520.0, -70000.0, np.inf, 2.0 ** -30, 3 * 2.0 ** -31, float.fromhex("0x1.234568p-20"),
    float.fromhex("0x1.000002p-8"), float.fromhex("0x1.fffffep-3"), 1.0 + 2.0 ** -23, 2.0 ** -20,
    float.fromhex("0x1.abcdeep5"), -float.fromhex("0x1.555554p-12"), 0.0,
]

# the other factor of each product: exact in fp16 and bf16, never zero
B_VALUES = np.array([0.5, 0.75, 1.0, 1.25, 1.5, -0.5, -0.75, -1.0, -1.25, -1.5], np.float32)


def _one_hot(specials, rows, k, seed, b_scale=1.0, n=48, b_values=B_VALUES):
    """A (rows x k): row i holds specials[i % len] at column (7 i) % k, zeros
    elsewhere; B (k x n): no zero entries.  Each C element is q(a) * q(b)."""
    g = np.random.Generator(np.random.PCG64(seed))
    a = np.zeros((rows, k), np.float32)
    for i in range(rows):
        a[i, (7 * i) % k] = np.float32(specials[i % len(specials)])
    b = (g.choice(b_values, size=(k, n)) * np.float32(b_scale)).astype(np.float32)
    return a, b


def _compare(got, ref, den, tol):
    """Non-finite results must match exactly (NaN for NaN, inf of the same
    sign for inf); finite ones within the normalised bar."""
    fin_ref = np.isfinite(ref)
    assert np.array_equal(np.isfinite(got), fin_ref), np.argwhere(np.isfinite(got) != fin_ref)[:5]
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    inf = np.isinf(ref)
    assert np.array_equal(got[inf], ref[inf])
    err = oracle.max_rel_err(got[fin_ref], ref[fin_ref], den[fin_ref])
    assert err <= tol, err
    return err


PATHS = {"onload": dict(prepass=-1), "pass": dict(prepass=1), "generic": dict(prepass=-1, force_generic_load=1)}


def _run(mode, q, a, b, path, transpose=False, extra=None, exps=(0, 0)):
    """C = A B (or, with transpose, C^T = B^T A^T: the specials in B) on one
    path; returns (gpu, ref, den) of the quantised-input problem."""
    opts = mpg.options(**PATHS[path], split_exp_a=exps[0], split_exp_b=exps[1], **(extra or {}))
    if transpose:
        a, b = np.ascontiguousarray(b.T), np.ascontiguousarray(a.T)
    m, k = a.shape
    n = b.shape[1]
    c = Case(m, n, k, mode, a=a[None], b=b[None], c0=np.zeros((1, m, n), np.float32),
             a_layout=mpg.ROW_MAJOR, b_layout=mpg.COL_MAJOR if transpose else mpg.ROW_MAJOR, opts=opts)
    c.run()
    got = c.result()[0]
    ref, den = oracle.gemm(a, b, None, 1.0, 0.0, q, q, exps[0], exps[1])
    return got, ref, den


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("side", ["A", "B"])
def test_fp16_conversion_edges(path, side):
    mpg.build()
    a, b = _one_hot(FP16_SPECIALS, 2 * len(FP16_SPECIALS), 40, 11)
    got, ref, den = _run(mpg.FP16_F32ACC, oracle.Q_FP16, a, b, path, transpose=(side == "B"))
    _compare(got, ref, den, TOL["q16"])
    # the overflow midpoint and beyond gave infinities, 65519.99 the largest finite value
    rows = {v: i for i, v in enumerate(FP16_SPECIALS) if not np.isnan(v)}
    col = (lambda i: got[i]) if side == "A" else (lambda i: got[:, i])
    assert np.all(np.isinf(col(rows[65520.0]))) and np.all(np.isfinite(col(rows[65519.99])))
    # fp16 subnormals were kept (gradual underflow), not flushed
    assert np.all(col(rows[2.0 ** -24]) != 0)


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("side", ["A", "B"])
def test_bf16_conversion_edges_large(path, side):
    mpg.build()
    a, b = _one_hot(BF16_LARGE, 2 * len(BF16_LARGE), 40, 12, b_values=B_VALUES[np.abs(B_VALUES) <= 1.0])
    got, ref, den = _run(mpg.BF16_F32ACC, oracle.Q_BF16, a, b, path, transpose=(side == "B"))
    _compare(got, ref, den, TOL["q16"])
    rows = {v: i for i, v in enumerate(BF16_LARGE) if not np.isnan(v)}
    col = (lambda i: got[i]) if side == "A" else (lambda i: got[:, i])
    assert np.all(np.isinf(col(rows[float.fromhex("0x1.ffp127")])))        # the midpoint ties up
    assert np.all(np.isfinite(col(rows[float.fromhex("0x1.fefffep127")])))


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("side", ["A", "B"])
def test_bf16_conversion_edges_subnormal(path, side):
    mpg.build()
    a, b = _one_hot(BF16_SMALL, 2 * len(BF16_SMALL), 40, 15, b_scale=2.0 ** 24)
    got, ref, den = _run(mpg.BF16_F32ACC, oracle.Q_BF16, a, b, path, transpose=(side == "B"))
    _compare(got, ref, den, TOL["q16"])
    rows = {v: i for i, v in enumerate(BF16_SMALL)}
    col = (lambda i: got[i]) if side == "A" else (lambda i: got[:, i])
    assert np.all(col(rows[2.0 ** -133]) != 0)                             # kept, not flushed


@pytest.mark.parametrize("path", list(PATHS))
@pytest.mark.parametrize("side", ["A", "B"])
@pytest.mark.parametrize("form", ["split3", "split3_plain", "split1"])
def test_split_edges(path, side, form):
    """The split at its documented range limit and where lo underflows:
    |x| >= 65520 gives hi = inf and lo = -inf, so the elements that product
    touches are NaN on the GPU as in the oracle; tiny values keep their lo
    half with the 2^11 scale and lose it without."""
    mpg.build()
    mode, q, extra = {"split3": (mpg.SPLIT_FP16_3CHAIN, oracle.Q_SPLIT3, None),
                      "split3_plain": (mpg.SPLIT_FP16_3CHAIN, oracle.Q_SPLIT1, dict(split_plain_lo=1)),
                      "split1": (mpg.SPLIT_FP16_1CHAIN, oracle.Q_SPLIT1, None)}[form]
    a, b = _one_hot(SPLIT_SPECIALS, 2 * len(SPLIT_SPECIALS), 40, 13)
    got, ref, den = _run(mode, q, a, b, path, transpose=(side == "B"), extra=extra)
    _compare(got, ref, den, TOL["q16"])
    rows = {v: i for i, v in enumerate(SPLIT_SPECIALS)}
    col = (lambda i: got[i]) if side == "A" else (lambda i: got[:, i])
    assert np.all(np.isnan(col(rows[65520.0]))) and np.all(np.isnan(col(rows[-70000.0])))
    assert np.all(np.isfinite(col(rows[65519.99])))
    tiny = col(rows[2.0 ** -30])
    if form == "split3":
        assert np.all(tiny != 0)          # lo = fp16(2^-30 * 2^11) = 2^-19 survives
    else:
        assert np.all(tiny == 0)          # hi = 0 and the plain lo fp16(2^-30) = 0


def test_split_range_with_operand_scale():
    """The precondition is on x * 2^s: with s = -2 the value 65520 * 3 = 196560
    splits finitely (196560 / 4 = 49140 < 65520), and 4 * 65520 does not."""
    mpg.build()
    specials = [196560.0, 4 * 65520.0, 1.0, -2.5]
    a, b = _one_hot(specials, 8, 16, 14)
    got, ref, den = _run(mpg.SPLIT_FP16_3CHAIN, oracle.Q_SPLIT3, a, b, "onload", exps=(-2, 0))
    _compare(got, ref, den, TOL["q16"])
    assert np.all(np.isfinite(got[0])) and np.all(np.isnan(got[1]))
