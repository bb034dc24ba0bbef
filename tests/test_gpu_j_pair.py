"""GPU parity of the CTA-pair kernel (cta_group::2, 256 x 256 tiles per
cluster of two CTAs) for 16-bit operands on the direct path: layouts, ragged
tails (including a second CTA whose rows all lie past m), batches, split-K,
16-bit output, the conversion pass's copies, and the full 8192^3 bf16 product
with beta = 0.5, each against the oracle."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic
from helpers import TOL, Case, sample_points

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR


def pair(**kw):
    return mpg.options(cta_pair=1, **kw)


def test_pair_smallest_tile():
    mpg.build()
    c = Case(256, 256, 64, mpg.BF16_F32ACC, in_dtype="bf16", dist="normal",
             opts=pair(wait_timeout_ns=200_000_000))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], eQ


@pytest.mark.parametrize("mode,dt", [(mpg.BF16_F32ACC, "bf16"), (mpg.FP16_F32ACC, "f16")])
@pytest.mark.parametrize("al,bl", [(R, R), (R, Cm), (Cm, R), (Cm, Cm)])
@pytest.mark.parametrize("m,n,k", [(300, 520, 200), (100, 260, 1000), (640, 96, 64)])
def test_pair_layouts_and_tails(mode, dt, al, bl, m, n, k):
    mpg.build()
    c = Case(m, n, k, mode, in_dtype=dt, a_layout=al, b_layout=bl, pad=(8, 8, 4), alpha=1.5, beta=-0.5,
             dist="normal", opts=pair())
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], eQ


def test_pair_batched_and_split_k():
    mpg.build()
    c = Case(200, 300, 512, mpg.BF16_F32ACC, batch=3, in_dtype="bf16", pad=(0, 8, 0), beta=0.25,
             dist="normal", opts=pair())
    c.run()
    assert c.errors()[1] <= TOL["q16"]
    c = Case(256, 256, 6144, mpg.FP16_F32ACC, in_dtype="f16", beta=1.0, dist="normal", opts=pair(splitk=4))
    c.run()
    assert c.errors()[1] <= TOL["q16"]


def test_pair_conversion_pass_copies():
    """fp32 operands rounded to fp16 by the separate pass, multiplied on pairs."""
    mpg.build()
    c = Case(384, 640, 320, mpg.FP16_F32ACC, in_dtype="f32", a_layout=Cm, dist="normal",
             opts=pair(prepass=1))
    c.run()
    assert c.errors()[1] <= TOL["q16"]


def test_pair_sixteen_bit_output():
    import torch
    mpg.build()
    m, n, k = 300, 272, 128
    a = synthetic.normal((m, k), 121)
    b = synthetic.normal((k, n), 122)
    A = torch.from_numpy(a).cuda().to(torch.bfloat16)
    B = torch.from_numpy(b).cuda().to(torch.bfloat16)
    C = torch.zeros((m, n), dtype=torch.float16, device="cuda")
    mpg.gemm(A, B, C, mode="bf16", opts=pair())
    got = C.float().cpu().numpy().astype(np.float64)
    ab = A.float().cpu().numpy()
    bb = B.float().cpu().numpy()
    ref, den = oracle.gemm(ab, bb)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))) - 10)
    assert np.all(np.abs(got - ref) <= ulp + TOL["q16"] * den)


def test_pair_full_size_bf16_8192_beta(capsys):
    mpg.build()
    n = 8192
    c = Case(n, n, n, mpg.BF16_F32ACC, in_dtype="bf16", dist="normal", alpha=1.0, beta=0.5,
             c0=synthetic.normal((n, n), synthetic.SEED_C0), opts=pair())
    c.run()
    C = c.result()
    rows, cols = sample_points(n, n, 3000, 83)
    ref, den = c.reference_points(oracle.Q_NONE, 0, rows, cols)
    err = oracle.max_rel_err(C[0][rows, cols], ref, den)
    r = np.array([0, 255, 256, 4095, 8191])
    refr, denr = oracle.gemm(c.a[0][r], c.b[0], c.c0[0][r], 1.0, 0.5)
    err_rows = oracle.max_rel_err(C[0][r], refr, denr)
    with capsys.disabled():
        print(f"\n[pair bf16 8192^3: sampled {err:.3e}, rows {err_rows:.3e}]")
    assert err <= TOL["q16"] and err_rows <= TOL["q16"]


# ---------------------------------------------------------------- split tail
@pytest.mark.parametrize("m,n,k,mode,dt,al,bl,batch", [
    (300, 520, 200, mpg.BF16_F32ACC, "bf16", R, R, 1),     # ragged k: 4 k-blocks, cut after 2
    (520, 300, 1000, mpg.FP16_F32ACC, "f16", Cm, R, 1),
    (200, 300, 520, mpg.BF16_F32ACC, "bf16", R, Cm, 3),
    (256, 256, 128, mpg.FP16_F32ACC, "f16", Cm, Cm, 2),    # two k-blocks: one each
    (300, 520, 200, mpg.TF32, "f32", R, Cm, 2),            # tf32: k-blocks of 32, cut after 3
])
def test_pair_split_tail_forced(m, n, k, mode, dt, al, bl, batch):
    """tail_split = 1 with fewer tiles than clusters: every tile is cut in
    two along K and the second half to finish adds the first's partial sums."""
    mpg.build()
    c = Case(m, n, k, mode, batch=batch, in_dtype=dt, a_layout=al, b_layout=bl, pad=(8, 0, 4), alpha=1.5,
             beta=-0.5, dist="normal", opts=pair(tail_split=1))
    c.run(exact_ws=True)
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    else:
        assert eQ <= TOL["q16"], eQ


def test_pair_split_tail_is_deterministic_and_sixteen_bit_output():
    import torch
    mpg.build()
    m, n, k = 300, 520, 700
    a = synthetic.normal((m, k), 131)
    b = synthetic.normal((k, n), 132)
    A = torch.from_numpy(a).cuda().to(torch.bfloat16)
    B = torch.from_numpy(b).cuda().to(torch.bfloat16)
    outs = []
    for _ in range(3):
        C = torch.zeros((m, n), dtype=torch.float32, device="cuda")
        mpg.gemm(A, B, C, mode="bf16", opts=pair(tail_split=1))
        outs.append(C.cpu().numpy())
    # the two halves meet in either order with the same sum
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))
    ref, den = oracle.gemm(A.float().cpu().numpy(), B.float().cpu().numpy())
    assert oracle.max_rel_err(outs[0], ref, den) <= TOL["q16"]
    # a 16-bit C: alpha * (half + half) + beta * C rounded once
    c0 = synthetic.uniform((m, n), 133).astype(np.float16)
    C16 = torch.from_numpy(c0).cuda()
    mpg.gemm(A, B, C16, alpha=0.75, beta=0.5, mode="bf16", opts=pair(tail_split=1))
    got = C16.float().cpu().numpy().astype(np.float64)
    ref, den = oracle.gemm(A.float().cpu().numpy(), B.float().cpu().numpy(), c0.astype(np.float32), 0.75, 0.5)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))) - 10)
    assert np.all(np.abs(got - ref) <= ulp + TOL["q16"] * den)


def test_pair_split_tail_needs_its_workspace():
    import torch
    mpg.build()
    A = torch.zeros((300, 200), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((200, 520), dtype=torch.bfloat16, device="cuda")
    C = torch.zeros((300, 520), dtype=torch.float32, device="cuda")
    st = mpg.gemm_raw(300, 520, 200, 1, A.data_ptr(), 200, 0, mpg.BF16, R, B.data_ptr(), 520, 0, mpg.BF16, R,
                      C.data_ptr(), 520, 0, 1.0, 0.0, mpg.BF16_F32ACC, opts=pair(tail_split=1), check=False)
    assert st == mpg.ERR_WORKSPACE and "split tail" in mpg.last_error()


def test_pair_split_tail_by_default_on_the_last_round(capsys):
    """2560 x 2560 x 8192 bf16: 100 tiles of 256 x 256, one full round on the
    device's clusters and a partial last round, which the library cuts in two
    along K by default (k >= 8192).  Against tail_split = -1 the tiles of the
    full round agree bit for bit, those of the last round differ in rounding
    only, and both products meet the oracle's bar on sampled points, among
    them 64 in every tile that was cut."""
    mpg.build()
    m = n = 2560
    k = 8192
    out = {}
    for ts in (0, -1):
        c = Case(m, n, k, mpg.BF16_F32ACC, in_dtype="bf16", dist="normal", beta=0.5, opts=pair(tail_split=ts))
        c.run()
        out[ts] = c.result()[0]
    tiles = m // 256
    cut = [(i, j) for i in range(tiles) for j in range(tiles)
           if not np.array_equal(out[0][256 * i:256 * (i + 1), 256 * j:256 * (j + 1)].view(np.uint32),
                                 out[-1][256 * i:256 * (i + 1), 256 * j:256 * (j + 1)].view(np.uint32))]
    # R tiles after W >= 1 full rounds of P clusters, 2R <= P: R <= 100 / 3
    assert 1 <= len(cut) and 3 * len(cut) <= tiles * tiles, len(cut)
    rows, cols = sample_points(m, n, 2000, 141)
    g = np.random.Generator(np.random.PCG64(142))
    for (i, j) in cut:
        rows = np.concatenate([rows, 256 * i + g.integers(0, 256, 64)])
        cols = np.concatenate([cols, 256 * j + g.integers(0, 256, 64)])
    ref, den = c.reference_points(oracle.Q_NONE, 0, rows, cols)
    errs = {ts: oracle.max_rel_err(out[ts][rows, cols], ref, den) for ts in out}
    with capsys.disabled():
        print(f"\n[split tail 2560^2 x 8192: {len(cut)} tiles cut; errors {errs}]")
    assert max(errs.values()) <= TOL["q16"], errs


# ---------------------------------------------------------------- tf32 pairs
@pytest.mark.parametrize("al,bl", [(R, Cm), (R, R), (Cm, Cm)])
@pytest.mark.parametrize("m,n,k,batch", [(300, 520, 200, 1), (520, 272, 1000, 2), (256, 256, 32, 1)])
def test_pair_tf32(al, bl, m, n, k, batch):
    """tf32 on CTA pairs (cta_group::2, kind::tf32), row-major A and column-
    major B on the direct path, other layouts through the transposed copies."""
    mpg.build()
    c = Case(m, n, k, mpg.TF32, batch=batch, a_layout=al, b_layout=bl, pad=(4, 8, 4), alpha=1.5, beta=-0.5,
             dist="normal", opts=pair())
    c.run(exact_ws=True)
    eR, _ = c.errors()
    assert eR <= TOL["tf32"], eR


@pytest.mark.parametrize("mode,dt", [(mpg.TF32, "f32"), (mpg.BF16_F32ACC, "bf16")])
def test_pair_matches_single_cta_bit_for_bit(mode, dt):
    """The pair form multiplies the same products in the same K order as
    the one-CTA form: the results agree bit for bit."""
    mpg.build()
    out = {}
    for cp in (1, -1):
        c = Case(520, 784, 1000, mode, in_dtype=dt, a_layout=R, b_layout=Cm, beta=0.5, dist="normal",
                 opts=mpg.options(cta_pair=cp))
        c.run(exact_ws=True)
        out[cp] = c.result()
    assert np.array_equal(out[1].view(np.uint32), out[-1].view(np.uint32))


@pytest.mark.parametrize("mode,dt,tail", [(mpg.BF16_F32ACC, "bf16", -1), (mpg.BF16_F32ACC, "bf16", 1),
                                          (mpg.TF32, "f32", -1), (mpg.TF32, "f32", 1)])
def test_pair_beta_zero_does_not_read_c(mode, dt, tail):
    """beta == 0 on CTA pairs, whole tiles and split tail: NaN in C must not
    leak into the result (C is written, never read)."""
    mpg.build()
    c = Case(300, 520, 400, mode, batch=2, in_dtype=dt, a_layout=R, b_layout=Cm, pad=(8, 8, 4), alpha=2.0,
             beta=0.0, dist="normal", opts=pair(tail_split=tail))
    c.C[:, :, :c.n] = float("nan")
    c.c0[...] = 0.0
    c.run(exact_ws=True)
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    else:
        assert eQ <= TOL["q16"], eQ


# ---------------------------------------------------------------- the split on pairs
@pytest.mark.parametrize("al,bl", [(R, R), (R, Cm), (Cm, R), (Cm, Cm)])
@pytest.mark.parametrize("m,n,k,batch,kw", [
    (512, 384, 1024, 1, {}),
    (300, 200, 700, 1, {}),                        # tails in both CTAs' rows and in the columns
    (260, 130, 1536, 2, dict(split_chunk_k=256)),  # batches, more K chunks
    (512, 256, 640, 1, dict(split_chunk_k=-1)),    # one chunk
    (384, 256, 512, 1, dict(split_plain_lo=1)),
])
def test_split3_pair_equals_single_cta(al, bl, m, n, k, batch, kw):
    """The three-chain split on the conversion pass's copies, on CTA pairs
    (256 x 128 tiles) and on single CTAs: the same products accumulated in
    the same K order and the same chunk folds, so the same bits; and within
    the split's bars against the oracle."""
    mpg.build()
    outs = []
    for cp in (1, -1):
        c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, batch=batch, a_layout=al, b_layout=bl, pad=(4, 8, 4),
                 alpha=1.0, beta=-0.5, dist="loguniform", seed=21, opts=mpg.options(prepass=1, cta_pair=cp, **kw))
        c.run()
        outs.append(c.result())
    assert np.array_equal(outs[0], outs[1])
    c.opts = mpg.options(prepass=1, cta_pair=1, **kw)
    q = oracle.Q_SPLIT1 if kw.get("split_plain_lo") else oracle.Q_SPLIT3
    for bi in range(batch):
        ref, den = c.reference(q, [bi])[0]
        assert oracle.max_rel_err(outs[0][bi], ref, den) <= TOL["q16"]
        refr, denr = c.reference(oracle.Q_NONE, [bi])[0]
        assert oracle.max_rel_err(outs[0][bi], refr, denr) <= TOL["split"]


def test_split3_pair_split_k_and_scales():
    """Split-K partial sums from the pair kernel, with operand exponents."""
    mpg.build()
    c = Case(256, 256, 8192, mpg.SPLIT_FP16_3CHAIN, alpha=2.0, dist="normal", seed=22,
             opts=mpg.options(prepass=1, cta_pair=1, splitk=3, split_exp_a=3, split_exp_b=-2))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)
