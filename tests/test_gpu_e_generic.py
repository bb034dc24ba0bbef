"""GPU: the generic-load path (converter warps read global memory directly),
used where TMA cannot describe the operands: leading dimensions whose byte
size is not a multiple of 16, unaligned base pointers, or on request."""
import pytest

import mixed_precision_matmul_gb300 as mpg
from helpers import TOL, Case

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR


@pytest.mark.parametrize("mode,dt", [
    (mpg.BF16_F32ACC, "bf16"), (mpg.FP16_F32ACC, "f16"), (mpg.TF32, "f32"),
    (mpg.FP16_F32ACC, "f32"), (mpg.BF16_F32ACC, "f32"),
    (mpg.SPLIT_FP16_3CHAIN, "f32"), (mpg.SPLIT_FP16_1CHAIN, "f32"),
])
@pytest.mark.parametrize("m,n,k,al,bl,pad,force", [
    (129, 131, 67, R, R, (2, 3, 1), 0),      # odd leading dims: TMA impossible
    (150, 100, 90, Cm, Cm, (3, 1, 0), 0),
    (128, 128, 64, R, Cm, (0, 0, 0), 1),     # aligned, generic on request
    (64, 200, 96, Cm, R, (0, 0, 0), 1),
])
def test_generic_parity(mode, dt, m, n, k, al, bl, pad, force):
    mpg.build()
    opts = mpg.options(force_generic_load=force)
    c = Case(m, n, k, mode, in_dtype=dt, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=0.5,
             dist="normal", opts=opts)
    c.run()
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    else:
        assert eQ <= TOL["q16"], (eR, eQ)
    if mode == mpg.SPLIT_FP16_3CHAIN:
        assert eR <= TOL["split"], eR


@pytest.mark.parametrize("mode,dt", [(mpg.BF16_F32ACC, "bf16"), (mpg.FP16_F32ACC, "f16"), (mpg.TF32, "f32")])
@pytest.mark.parametrize("m,n,k,al,bl,pad,batch", [
    (300, 260, 201, R, Cm, (0, 1, 3), 1),    # A's rows of 201 elements: A copied; B too (ldb 202)
    (300, 260, 200, R, Cm, (0, 3, 0), 1),    # only B unaligned (ldb 203)
    (200, 130, 130, R, Cm, (1, 0, 2), 3),    # batches with odd strides (lda 131)
])
def test_unaligned_operands_copied_to_the_tma_path(mode, dt, m, n, k, al, bl, pad, batch):
    """With the workspace the exact query asks for, operands TMA cannot
    describe are copied to aligned lines and multiplied on the direct path."""
    mpg.build()
    c = Case(m, n, k, mode, in_dtype=dt, a_layout=al, b_layout=bl, pad=pad, alpha=1.25, beta=-0.5,
             dist="normal", batch=batch)
    ws_plain = mpg.workspace_size(m, n, k, batch, mode)
    c.run(exact_ws=True)
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"], eR
    else:
        assert eQ <= TOL["q16"], (eR, eQ)
    ws_exact = mpg.workspace_size_ex(m, n, k, batch, c.A.data_ptr(), c.lda, c.A.stride(0) if batch > 1 else 0,
                                     {"bf16": mpg.BF16, "f16": mpg.F16, "f32": mpg.F32}[dt], al, c.B.data_ptr(),
                                     c.ldb, c.B.stride(0) if batch > 1 else 0,
                                     {"bf16": mpg.BF16, "f16": mpg.F16, "f32": mpg.F32}[dt], bl, mode)
    assert ws_exact > ws_plain     # room for the copies was asked for


@pytest.mark.parametrize("m,n,k,al,bl,pad,batch", [
    (300, 260, 200, R, R, (0, 0, 0), 1),     # B row-major: transposed copy of B
    (300, 260, 200, Cm, Cm, (0, 0, 0), 1),   # A column-major: transposed copy of A
    (257, 131, 99, Cm, R, (1, 3, 2), 2),     # both transposed, odd leading dims, batches
])
def test_tf32_operands_transposed_to_the_direct_path(m, n, k, al, bl, pad, batch):
    """tf32 tiles are K-major: with the exact workspace, a column-major A or a
    row-major B is copied transposed and the direct tf32 path multiplies it."""
    mpg.build()
    c = Case(m, n, k, mpg.TF32, in_dtype="f32", a_layout=al, b_layout=bl, pad=pad, alpha=0.75, beta=0.5,
             dist="normal", batch=batch)
    c.run(exact_ws=True)
    eR, _ = c.errors()
    assert eR <= TOL["tf32"], eR
    ws_exact = mpg.workspace_size_ex(m, n, k, batch, c.A.data_ptr(), c.lda, c.A.stride(0) if batch > 1 else 0,
                                     mpg.F32, al, c.B.data_ptr(), c.ldb, c.B.stride(0) if batch > 1 else 0,
                                     mpg.F32, bl, mpg.TF32)
    assert ws_exact > mpg.workspace_size(m, n, k, batch, mpg.TF32)
