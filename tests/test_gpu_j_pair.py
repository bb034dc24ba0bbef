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
