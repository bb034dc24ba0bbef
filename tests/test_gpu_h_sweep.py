"""GPU: a seeded random sweep over the product's parameter space — precision
mode, storage type, both layouts, ragged sizes, leading-dimension padding,
batches, alpha/beta, tile width, forced generic loads, split-K — each case
checked against the oracle with the bar of its mode."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
from helpers import TOL, Case

pytestmark = pytest.mark.gpu

MODES = [(mpg.FP16_F32ACC, "f32"), (mpg.FP16_F32ACC, "f16"), (mpg.BF16_F32ACC, "f32"),
         (mpg.BF16_F32ACC, "bf16"), (mpg.TF32, "f32"), (mpg.SPLIT_FP16_3CHAIN, "f32"),
         (mpg.SPLIT_FP16_1CHAIN, "f32"), (mpg.FP32_FFMA, "f32"), (mpg.SPLIT_A_FP16_2CHAIN, "f32"),
         (mpg.SPLIT_FP16_4CHAIN, "f32")]


def _cases(n=64, seed=20251):
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for i in range(n):
        mode, dt = MODES[i % len(MODES)]
        m = int(g.integers(1, 300))
        nn = int(g.integers(1, 300))
        k = int(g.integers(1, 400))
        batch = int(g.choice([1, 1, 1, 2, 3]))
        al = int(g.integers(0, 2))
        bl = int(g.integers(0, 2))
        pad = tuple(int(x) for x in g.choice([0, 0, 1, 3, 8], size=3))
        alpha = float(g.choice([1.0, -0.5, 2.0]))
        beta = float(g.choice([0.0, 0.0, 1.0, -0.75]))
        force = int(g.random() < 0.2)
        splitk = int(g.choice([0, 0, 0, 2, 3])) if mode != mpg.FP32_FFMA else 0
        prepass = int(g.random() < 0.3 and dt == "f32" and mode not in (mpg.TF32, mpg.FP32_FFMA))
        out.append((i, mode, dt, m, nn, k, batch, al, bl, pad, alpha, beta, force, splitk, prepass))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: f"c{c[0]}")
def test_random_case(case):
    i, mode, dt, m, n, k, batch, al, bl, pad, alpha, beta, force, splitk, prepass = case
    mpg.build()
    opts = mpg.options(force_generic_load=force, splitk=splitk, prepass=prepass)
    c = Case(m, n, k, mode, batch=batch, in_dtype=dt, a_layout=al, b_layout=bl, pad=pad,
             alpha=alpha, beta=beta, seed=i, dist="normal", opts=opts)
    c.run()
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    elif mode == mpg.FP32_FFMA:
        assert eR <= TOL["q16"], eR
    else:
        assert eQ <= TOL["q16"], (eR, eQ)
    if mode in (mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_4CHAIN):
        assert eR <= TOL["split"], eR


PAIR_MODES = [(mpg.FP16_F32ACC, "f16"), (mpg.BF16_F32ACC, "bf16"), (mpg.TF32, "f32"), (mpg.FP16_F32ACC, "f32"),
              (mpg.BF16_F32ACC, "f32")]


def _pair_cases(n=30, seed=20252):
    """Cases that take the CTA-pair kernel (cta_pair = 1) whenever their path
    allows it, with the split tail forced, automatic or off."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for i in range(n):
        mode, dt = PAIR_MODES[i % len(PAIR_MODES)]
        m = int(g.integers(1, 700))
        nn = int(g.integers(1, 700))
        k = int(g.integers(1, 700))
        batch = int(g.choice([1, 1, 2, 3]))
        al = int(g.integers(0, 2))
        bl = int(g.integers(0, 2))
        pad = tuple(int(x) for x in g.choice([0, 0, 1, 8], size=3))
        alpha = float(g.choice([1.0, -0.5, 2.0]))
        beta = float(g.choice([0.0, 1.0, -0.75]))
        tail = int(g.choice([-1, 0, 1]))
        prepass = int(dt == "f32" and mode != mpg.TF32 and g.random() < 0.5)
        out.append((i, mode, dt, m, nn, k, batch, al, bl, pad, alpha, beta, tail, prepass))
    return out


@pytest.mark.parametrize("case", _pair_cases(), ids=lambda c: f"p{c[0]}")
def test_random_pair_case(case):
    i, mode, dt, m, n, k, batch, al, bl, pad, alpha, beta, tail, prepass = case
    mpg.build()
    opts = mpg.options(cta_pair=1, tail_split=tail, prepass=prepass)
    c = Case(m, n, k, mode, batch=batch, in_dtype=dt, a_layout=al, b_layout=bl, pad=pad,
             alpha=alpha, beta=beta, seed=100 + i, dist="normal", opts=opts)
    c.run(exact_ws=True)
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    else:
        assert eQ <= TOL["q16"], (eR, eQ)


SPLIT_MODES = [mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_1CHAIN,
               mpg.SPLIT_A_FP16_2CHAIN, mpg.SPLIT_FP16_4CHAIN]


def _split_cases(n=48, seed=20253):
    """The split modes with their own options drawn at random: the unscaled
    lo (split_plain_lo), the shared lo accumulator (split_lo_shared), the K
    chunk, per-operand power-of-two scales, the conversion pass or not, CTA
    pairs on the pass's copies, split-K, and C widths that do and do not
    allow the TMA-store epilogue (n % 4, beta)."""
    g = np.random.Generator(np.random.PCG64(seed))
    out = []
    for i in range(n):
        mode = SPLIT_MODES[i % len(SPLIT_MODES)]
        m = int(g.integers(1, 400))
        nn = int(g.integers(1, 75)) * 4 - int(g.choice([0, 0, 1, 3]))
        k = int(g.integers(1, 1200))
        batch = int(g.choice([1, 1, 2, 3]))
        al, bl = int(g.integers(0, 2)), int(g.integers(0, 2))
        pad = tuple(int(x) for x in g.choice([0, 0, 0, 1, 4], size=3))
        alpha = float(g.choice([1.0, -0.5, 2.0]))
        beta = float(g.choice([0.0, 0.0, 1.0, -0.75]))
        s3 = mode == mpg.SPLIT_FP16_3CHAIN
        opts = dict(
            split_plain_lo=int(s3 and g.random() < 0.3),
            split_lo_shared=int(s3 and g.random() < 0.4),
            split_chunk_k=int(g.choice([0, 0, -1, 64, 192, 512])),
            split_exp_a=0, split_exp_b=0,
            splitk=int(g.choice([0, 0, 2, 3])),
            prepass=int(g.choice([-1, 0, 1])),
            cta_pair=int(g.choice([0, 0, 1])),
            force_generic_load=int(g.random() < 0.15),
        )
        opts["split_exp_a"], opts["split_exp_b"] = [(0, 0), (0, 0), (-2, 3), (4, -1)][int(g.integers(0, 4))]
        dist = str(g.choice(["normal", "normal", "loguniform"]))
        out.append((i, mode, m, nn, k, batch, al, bl, pad, alpha, beta, opts, dist))
    return out


@pytest.mark.parametrize("case", _split_cases(), ids=lambda c: f"s{c[0]}")
def test_random_split_options(case):
    import oracle
    i, mode, m, n, k, batch, al, bl, pad, alpha, beta, kw, dist = case
    mpg.build()
    c = Case(m, n, k, mode, batch=batch, a_layout=al, b_layout=bl, pad=pad, alpha=alpha, beta=beta,
             seed=100 + i, dist=dist, opts=mpg.options(**kw))
    c.run()
    got = c.result()
    plain = mode == mpg.SPLIT_FP16_1CHAIN or kw["split_plain_lo"]
    q = {mpg.SPLIT_FP16_3CHAIN: oracle.Q_SPLIT1 if plain else oracle.Q_SPLIT3,
         mpg.SPLIT_FP16_1CHAIN: oracle.Q_SPLIT1, mpg.SPLIT_A_FP16_2CHAIN: oracle.Q_SPLIT3,
         mpg.SPLIT_FP16_4CHAIN: oracle.Q_SPLIT4}[mode]
    qb = oracle.Q_FP16 if mode == mpg.SPLIT_A_FP16_2CHAIN else None
    eQ = max(oracle.max_rel_err(got[bi], *r) for bi, r in enumerate(c.reference(q, qb=qb)))
    assert eQ <= TOL["q16"], eQ
    if mode in (mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_4CHAIN) and not plain:
        eR = max(oracle.max_rel_err(got[bi], *r) for bi, r in enumerate(c.reference(oracle.Q_NONE)))
        assert eR <= TOL["split"], eR
