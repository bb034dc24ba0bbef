"""GPU: fp32 operands converted on load (TMA staging + converter warps):
fp16 / bf16 rounding and the hi/lo split in its three-chain and one-chain
forms, against both oracle modes."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
from helpers import TOL, Case, sample_points

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR
SHAPES = [
    (128, 128, 32, R, R, (0, 0, 0), 0),
    (128, 128, 32, R, Cm, (0, 0, 0), 0),
    (128, 128, 32, Cm, R, (0, 0, 0), 0),
    (128, 128, 32, Cm, Cm, (0, 0, 0), 0),
    (333, 270, 150, R, R, (4, 4, 4), 0),       # ragged tails, padded
    (140, 300, 72, Cm, R, (8, 0, 4), 64),      # 64-wide tiles
    (100, 100, 600, R, Cm, (0, 4, 0), 128),    # long K
]


@pytest.mark.parametrize("mode", [mpg.FP16_F32ACC, mpg.BF16_F32ACC])
@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES)
def test_round_on_load_parity(mode, m, n, k, al, bl, pad, tile_n):
    mpg.build()
    opts = mpg.options(tile_n=tile_n) if tile_n else None
    c = Case(m, n, k, mode, a_layout=al, b_layout=bl, pad=pad, alpha=0.5, beta=1.5, opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)


@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES)
def test_split3_parity(m, n, k, al, bl, pad, tile_n):
    mpg.build()
    opts = mpg.options(tile_n=tile_n) if tile_n else None
    c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=-1.0,
             opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)
    assert eR <= TOL["split"], (eR, eQ)


@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES[:5])
def test_split1_parity(m, n, k, al, bl, pad, tile_n):
    mpg.build()
    c = Case(m, n, k, mpg.SPLIT_FP16_1CHAIN, a_layout=al, b_layout=bl, pad=pad)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)


def test_split_operand_scale():
    """Operands far below fp16's normal range need the power-of-two operand
    scale; with it the split stays within the fp32-input error bar."""
    mpg.build()
    import synthetic
    a = synthetic.uniform((1, 200, 300), 71, 0.0, 1e-5)   # ~softmax-sized values
    b = synthetic.normal((1, 300, 130), 72)
    opts = mpg.options(split_exp_a=14)
    c = Case(200, 130, 300, mpg.SPLIT_FP16_3CHAIN, a=a, b=b, opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)


@pytest.mark.parametrize("mode", [mpg.FP16_F32ACC, mpg.BF16_F32ACC, mpg.SPLIT_FP16_3CHAIN,
                                  mpg.SPLIT_FP16_1CHAIN])
@pytest.mark.parametrize("tile_n", [64, 128])
def test_many_tiles_per_persistent_cta(mode, tile_n):
    """2048 x 2048 tiles over 152 persistent CTAs: every CTA walks many tiles
    through the staging / operand rings and both accumulator buffers (the
    regime where a staging buffer handed back to TMA too early showed up)."""
    import numpy as np
    import oracle
    from helpers import MODE_Q
    mpg.build()
    c = Case(2048, 2048, 512, mode, b_layout=Cm, opts=mpg.options(tile_n=tile_n))
    c.run()
    C = c.result()
    rows = np.array([0, 1, 127, 128, 1000, 1500, 2047])
    ref, den = oracle.gemm(c.a[0][rows], c.b[0], c.c0[0][rows], 1.0, 0.0, MODE_Q[mode], MODE_Q[mode])
    assert oracle.max_rel_err(C[0][rows], ref, den) <= TOL["q16"]


@pytest.mark.parametrize("chunk_k", [-1, 32, 96, 256])
@pytest.mark.parametrize("tile_n", [64, 128])
def test_split3_chunked_accumulation(chunk_k, tile_n):
    """The three-chain split folds each K chunk into an fp32 running sum kept
    in TMEM: many small chunks, chunks not dividing K, and a single chunk
    (no folding) must all meet both bars."""
    mpg.build()
    opts = mpg.options(tile_n=tile_n, split_chunk_k=chunk_k)
    c = Case(300, 260, 700, mpg.SPLIT_FP16_3CHAIN, b_layout=Cm, alpha=1.5, beta=0.5, opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)


@pytest.mark.parametrize("mode", [mpg.FP16_F32ACC, mpg.BF16_F32ACC])
@pytest.mark.parametrize("m,n,k,al,bl,pad", [
    (128, 256, 64, R, Cm, (0, 0, 0)),
    (300, 520, 100, R, R, (4, 4, 4)),
    (257, 700, 96, Cm, Cm, (7, 8, 0)),      # lda 264, ldb 104: TMA-aligned pitches
])
def test_round_on_load_256_wide_tiles(mode, m, n, k, al, bl, pad):
    mpg.build()
    c = Case(m, n, k, mode, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=0.5,
             opts=mpg.options(tile_n=256))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)


@pytest.mark.parametrize("mode", [mpg.FP16_F32ACC, mpg.BF16_F32ACC, mpg.SPLIT_FP16_3CHAIN,
                                  mpg.SPLIT_FP16_1CHAIN])
@pytest.mark.parametrize("m,n,k,al,bl,pad,batch", [
    (128, 128, 64, R, Cm, (0, 0, 0), 1),
    (333, 270, 150, R, R, (4, 4, 4), 1),
    (140, 300, 72, Cm, R, (3, 1, 4), 2),       # odd pitches: the copies are re-pitched for TMA
    (100, 100, 700, R, Cm, (0, 4, 0), 1),      # split-K as well
])
def test_separate_conversion_pass(mode, m, n, k, al, bl, pad, batch):
    """Operands converted by the separate pass into the workspace, then the
    direct TMA path: same bars as the on-the-fly conversion."""
    mpg.build()
    c = Case(m, n, k, mode, batch=batch, a_layout=al, b_layout=bl, pad=pad, alpha=1.25, beta=-0.5,
             opts=mpg.options(prepass=1))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)
    if mode == mpg.SPLIT_FP16_3CHAIN:
        assert eR <= TOL["split"], eR


def test_separate_conversion_pass_operand_scale():
    import synthetic
    mpg.build()
    a = synthetic.uniform((1, 200, 300), 71, 0.0, 1e-5)
    b = synthetic.normal((1, 300, 130), 72)
    c = Case(200, 130, 300, mpg.SPLIT_FP16_3CHAIN, a=a, b=b, opts=mpg.options(split_exp_a=14, prepass=1))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)


def test_separate_conversion_pass_needs_workspace():
    import torch
    mpg.build()
    m = n = k = 256
    A = torch.zeros((m, k), device="cuda")
    B = torch.zeros((k, n), device="cuda")
    C = torch.zeros((m, n), device="cuda")
    st = mpg.gemm_raw(m, n, k, 1, A.data_ptr(), k, 0, mpg.F32, R, B.data_ptr(), n, 0, mpg.F32, R, C.data_ptr(), n,
                      0, 1.0, 0.0, mpg.SPLIT_FP16_3CHAIN, opts=mpg.options(prepass=1), check=False)
    assert st == mpg.ERR_WORKSPACE
    assert mpg.workspace_size(m, n, k, 1, mpg.SPLIT_FP16_3CHAIN, mpg.options(prepass=1)) >= 4 * (m * k + k * n)


@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES)
@pytest.mark.parametrize("prepass", [0, 1])
def test_split_a_two_chain_parity(m, n, k, al, bl, pad, tile_n, prepass):
    """The Volta page's form: A split into hi and lo, B rounded to fp16, the
    hi and lo products in separate chains.  Against the problem on the inputs
    as quantised (A = hi + lo, B = fp16(B))."""
    mpg.build()
    opts = mpg.options(tile_n=tile_n if not prepass else 0, prepass=prepass)
    c = Case(m, n, k, mpg.SPLIT_A_FP16_2CHAIN, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=0.5,
             opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)


@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES)
@pytest.mark.parametrize("prepass", [0, 1])
def test_split_four_chain_parity(m, n, k, al, bl, pad, tile_n, prepass):
    """hi*hi, hi*lo, lo*hi and lo*lo in four chains (128 x 64 tiles)."""
    mpg.build()
    c = Case(m, n, k, mpg.SPLIT_FP16_4CHAIN, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=-0.5,
             opts=mpg.options(prepass=prepass))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)


@pytest.mark.parametrize("mode,q", [(mpg.FP16_F32ACC, oracle.Q_FP16), (mpg.BF16_F32ACC, oracle.Q_BF16)])
def test_fp16_modes_on_fp32_take_the_pass_with_the_exact_workspace(mode, q):
    """2048 x 2048 x 1024 (2^32 multiply-adds): with the workspace the exact
    query asks for, fp32 operands are converted by the separate pass; the
    result equals the on-load conversion's within the mode's bar."""
    import torch
    mpg.build()
    m = n = 2048
    k = 1024
    c = Case(m, n, k, mode, b_layout=Cm, alpha=1.0, beta=0.5, dist="normal")
    c.run(exact_ws=True)
    rows, cols = sample_points(m, n, 1500, 91)
    ref, den = c.reference_points(q, 0, rows, cols)
    err = oracle.max_rel_err(c.result()[0][rows, cols], ref, den)
    assert err <= TOL["q16"], err
    # the torch wrapper sizes its workspace with the exact query
    A = torch.from_numpy(c.a[0]).cuda()
    B = torch.from_numpy(c.b[0]).cuda()
    C = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    mpg.gemm(A, B, C, mode=mode)
    torch.cuda.synchronize()
    ref, den = c.reference_points(q, 0, rows, cols)
    ref0 = ref - 0.5 * c.c0[0][rows, cols].astype(np.float64)   # the wrapper call used beta = 0
    den0 = den - 0.5 * np.abs(c.c0[0][rows, cols].astype(np.float64))
    assert oracle.max_rel_err(C.cpu().numpy()[rows, cols], ref0, den0) <= TOL["q16"]


@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES[:5])
@pytest.mark.parametrize("prepass", [-1, 1])
def test_split3_plain_lo_parity(m, n, k, al, bl, pad, tile_n, prepass):
    """The three-chain split with the plain lo = fp16(x - hi): its quantised
    problem is the one-chain form's (hi, plain lo, three products)."""
    mpg.build()
    opts = mpg.options(split_plain_lo=1, prepass=prepass, tile_n=tile_n)
    c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=-1.0, opts=opts)
    c.run()
    C = c.result()
    ref, den = c.reference(oracle.Q_SPLIT1)[0]
    assert oracle.max_rel_err(C[0], ref, den) <= TOL["q16"]


def test_chain_count_alone_on_identical_operands():
    """Three chains against one on bit-identical operands (plain lo, one K
    chunk, same operand scale): the only difference is whether the lo
    products have accumulators of their own ("qsa_prompt_attn ...", "The
    fix").  On log-uniform magnitudes the separate chains are closer to the
    quantised problem and to the fp32-input problem."""
    mpg.build()
    m = n = 384
    k = 4096
    errs = {}
    for name, mode, extra in (("3chain", mpg.SPLIT_FP16_3CHAIN, dict(split_plain_lo=1, split_chunk_k=-1)),
                              ("1chain", mpg.SPLIT_FP16_1CHAIN, {})):
        c = Case(m, n, k, mode, dist="loguniform", seed=5, opts=mpg.options(prepass=-1, **extra))
        c.run()
        C = c.result()[0]
        refQ, denQ = c.reference(oracle.Q_SPLIT1)[0]
        refR, denR = c.reference(oracle.Q_NONE)[0]
        errs[name] = (oracle.max_rel_err(C, refQ, denQ), oracle.max_rel_err(C, refR, denR))
    assert errs["3chain"][0] <= TOL["q16"], errs
    assert errs["3chain"][0] < errs["1chain"][0], errs
    assert errs["3chain"][1] < errs["1chain"][1], errs


@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", SHAPES[:6])
@pytest.mark.parametrize("prepass", [-1, 1])
def test_split3_shared_lo_accumulator_parity(m, n, k, al, bl, pad, tile_n, prepass):
    """Two accumulators (hh, and hl + lh together): the same quantised
    problem as the three chains, within the same bars."""
    mpg.build()
    opts = mpg.options(split_lo_shared=1, prepass=prepass, tile_n=tile_n)
    c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=-1.0, opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)


def test_split3_shared_lo_many_tiles_both_buffers():
    """1024 x 4096 x 128 on 128 x 128 tiles: 256 tiles over the persistent
    CTAs, every CTA cycling through both accumulator buffers."""
    mpg.build()
    c = Case(1024, 4096, 128, mpg.SPLIT_FP16_3CHAIN, b_layout=Cm, dist="normal", seed=3,
             opts=mpg.options(split_lo_shared=1, prepass=-1))
    c.run()
    C = c.result()
    rows, cols = sample_points(1024, 4096, 3000, 33)
    ref, den = c.reference_points(oracle.Q_NONE, 0, rows, cols)
    assert oracle.max_rel_err(C[0][rows, cols], ref, den) <= TOL["split"]
    refq, denq = c.reference_points(oracle.Q_SPLIT3, 0, rows, cols)
    assert oracle.max_rel_err(C[0][rows, cols], refq, denq) <= TOL["q16"]


def test_split3_shared_lo_falls_back_beyond_one_chunk():
    """k above the accumulation chunk: the option leaves the three chains,
    so the result is the default's bit for bit."""
    mpg.build()
    outs = []
    for shared in (0, 1):
        c = Case(200, 136, 1200, mpg.SPLIT_FP16_3CHAIN, seed=4, opts=mpg.options(split_lo_shared=shared))
        c.run()
        outs.append(c.result())
    assert np.array_equal(outs[0], outs[1])
