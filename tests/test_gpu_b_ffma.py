"""GPU: the plain fp32 FFMA comparator against the oracle (mode R)."""
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
