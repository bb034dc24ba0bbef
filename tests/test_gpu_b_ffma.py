"""GPU: the plain fp32 FFMA comparator against the oracle (mode R)."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
from helpers import Case

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,n,k,al,bl,pad", [
    (128, 128, 64, mpg.ROW_MAJOR, mpg.ROW_MAJOR, (0, 0, 0)),
    (301, 259, 131, mpg.ROW_MAJOR, mpg.ROW_MAJOR, (3, 5, 7)),
    (77, 190, 45, mpg.COL_MAJOR, mpg.COL_MAJOR, (1, 2, 3)),
    (1, 1, 1, mpg.ROW_MAJOR, mpg.COL_MAJOR, (0, 0, 0)),
])
def test_ffma_parity(m, n, k, al, bl, pad):
    mpg.build()
    c = Case(m, n, k, mpg.FP32_FFMA, a_layout=al, b_layout=bl, pad=pad, alpha=0.75, beta=-0.5)
    c.run()
    eR, _ = c.errors()
    assert eR <= 1e-5, eR


@pytest.mark.parametrize("m,n,k,batch,al,bl,pad,beta", [
    (128, 128, 64, 1, mpg.ROW_MAJOR, mpg.ROW_MAJOR, (0, 0, 0), 0.0),
    (301, 259, 131, 1, mpg.ROW_MAJOR, mpg.ROW_MAJOR, (3, 5, 7), -0.5),
    (77, 190, 45, 1, mpg.COL_MAJOR, mpg.COL_MAJOR, (1, 2, 3), 0.25),
    (333, 260, 517, 2, mpg.ROW_MAJOR, mpg.COL_MAJOR, (0, 0, 4), 1.0),
    (256, 384, 512, 1, mpg.COL_MAJOR, mpg.ROW_MAJOR, (0, 0, 0), 0.0),
    (1, 1, 1, 1, mpg.ROW_MAJOR, mpg.COL_MAJOR, (0, 0, 0), 2.0),
])
def test_ffma_bit_exact_fma_chain(m, n, k, batch, al, bl, pad, beta):
    """Every element is the oracle's fp32 fmaf chain (k ascending, then the
    alpha / beta epilogue) bit for bit: aligned operands (vector loads) and
    padded ones (element loads), every layout, tails in M, N and K."""
    import oracle
    mpg.build()
    c = Case(m, n, k, mpg.FP32_FFMA, batch=batch, a_layout=al, b_layout=bl, pad=pad, alpha=0.75, beta=beta,
             dist="normal", seed=5)
    c.run()
    got = c.result()
    for bi in range(batch):
        ref = oracle.gemm_fma_chain_f32(c.a[bi], c.b[bi], c.c0[bi], 0.75, beta)
        assert np.array_equal(got[bi].view(np.uint32), ref.view(np.uint32)), \
            (bi, int(np.sum(got[bi].view(np.uint32) != ref.view(np.uint32))))
