"""GPU: the one-CTA epilogue's TMA stores.  Where C is fp32, beta is 0 and
a row of C is a whole number of 16-byte chunks (n % 4 == 0, aligned base,
ldc and batch stride), each epilogue warp stores its 32 x 32 block with one
tiled TMA store from its swizzled staging buffer; split-K partial sums go
the same way.  Checked against the oracle with C's padding columns as
canaries (no store may touch them), and bit for bit against the register
stores that a C one element off 16-byte alignment takes."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
from helpers import SENTINEL_BITS, TOL, Case

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR

CASES = [
    # mode, in_dtype, m, n, k, batch, pad of C, options
    (mpg.BF16_F32ACC, "bf16", 300, 68, 256, 1, 0, {}),
    (mpg.BF16_F32ACC, "bf16", 300, 69, 256, 1, 3, {}),      # ragged row: register stores
    (mpg.FP16_F32ACC, "f16", 257, 200, 192, 3, 4, dict(cta_pair=-1)),
    (mpg.TF32, "f32", 200, 72, 130, 2, 0, {}),
    (mpg.SPLIT_FP16_3CHAIN, "f32", 333, 140, 150, 1, 4, dict(prepass=-1)),
    (mpg.SPLIT_FP16_3CHAIN, "f32", 333, 140, 150, 1, 4, dict(prepass=-1, split_lo_shared=1)),
    (mpg.SPLIT_FP16_3CHAIN, "f32", 256, 128, 4096, 1, 0, dict(splitk=3)),   # partial sums by TMA
    (mpg.SPLIT_FP16_3CHAIN, "f32", 256, 130, 4096, 1, 2, dict(splitk=3)),   # n % 4 != 0: register stores
]


def _col_major_b(mode):
    return Cm if mode == mpg.TF32 else R


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"m{c[0]}_{c[3]}x{c[4]}x{c[5]}_b{c[6]}")
def test_tma_store_epilogue_against_oracle(case):
    mode, dt, m, n, k, batch, pc, kw = case
    mpg.build()
    c = Case(m, n, k, mode, batch=batch, in_dtype=dt, b_layout=_col_major_b(mode), pad=(0, 0, pc),
             alpha=0.75, beta=0.0, dist="normal", seed=7, opts=mpg.options(**kw))
    c.run()
    eR, eQ = c.errors()      # result() also checks every padding column of C
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    else:
        assert eQ <= TOL["q16"], (eR, eQ)


@pytest.mark.parametrize("mode,dt,kw", [(mpg.BF16_F32ACC, "bf16", {}), (mpg.TF32, "f32", {}),
                                        (mpg.SPLIT_FP16_3CHAIN, "f32", dict(prepass=-1))])
def test_tma_store_equals_register_stores_bit_for_bit(mode, dt, kw):
    """The same product into a 16-byte aligned C (TMA stores) and into a C
    that starts one float later (register stores): identical bits."""
    import torch
    mpg.build()
    m, n, k = 300, 264, 200
    c = Case(m, n, k, mode, in_dtype=dt, b_layout=_col_major_b(mode), alpha=-1.25, beta=0.0, dist="normal",
             seed=8, opts=mpg.options(**kw))
    c.run()
    aligned = c.result()[0]
    buf = torch.empty(m * n + 1, dtype=torch.float32, device="cuda")
    buf.view(torch.int32).fill_(int(SENTINEL_BITS.view(np.int32)))
    Cu = buf[1:]                                     # 4-byte aligned only
    mpg.gemm_raw(m, n, k, 1, c.A.data_ptr(), c.lda, 0, {"f32": mpg.F32, "bf16": mpg.BF16}[dt], c.a_layout,
                 c.B.data_ptr(), c.ldb, 0, {"f32": mpg.F32, "bf16": mpg.BF16}[dt], c.b_layout, Cu.data_ptr(), n, 0,
                 -1.25, 0.0, mode, 0, 0, 0, mpg.options(**kw))
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    out = buf.cpu().numpy()
    assert out[:1].view(np.uint32)[0] == SENTINEL_BITS
    assert np.array_equal(out[1:].reshape(m, n).view(np.uint32), aligned.view(np.uint32))
