"""GPU: the degenerate cases of C = alpha*A*B + beta*C (BLAS conventions, the
pages being silent): k == 0 gives beta*C; alpha == 0 reads neither A nor B;
beta == 0 never reads C; empty problems touch nothing; batch strides that are
not packed; a single-element product."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
from helpers import TOL, Case

pytestmark = pytest.mark.gpu

MODES = [mpg.FP16_F32ACC, mpg.BF16_F32ACC, mpg.TF32, mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_1CHAIN,
         mpg.FP32_FFMA]


def _raw(c, m=None, n=None, k=None, batch=None, A=None, B=None, alpha=None, beta=None):
    return mpg.gemm_raw(c.m if m is None else m, c.n if n is None else n, c.k if k is None else k,
                        c.batch if batch is None else batch,
                        c.A.data_ptr() if A is None else A, c.lda, 0, mpg.F32, c.a_layout,
                        c.B.data_ptr() if B is None else B, c.ldb, 0, mpg.F32, c.b_layout,
                        c.C.data_ptr(), c.ldc, 0, c.alpha if alpha is None else alpha,
                        c.beta if beta is None else beta, c.mode, check=False)


@pytest.mark.parametrize("mode", MODES)
def test_k_zero_scales_c(mode):
    mpg.build()
    c = Case(70, 50, 8, mode, pad=(0, 0, 3))
    assert _raw(c, k=0, alpha=2.0, beta=-0.5) == mpg.OK
    assert np.array_equal(c.result()[0], np.float32(-0.5) * c.c0[0])


@pytest.mark.parametrize("mode", MODES)
def test_alpha_zero_reads_no_operand(mode):
    mpg.build()
    c = Case(70, 50, 40, mode, pad=(0, 0, 3))
    # NULL operands: the call must not touch them
    assert _raw(c, A=0, B=0, alpha=0.0, beta=0.25) == mpg.OK
    assert np.array_equal(c.result()[0], np.float32(0.25) * c.c0[0])
    # beta == 0 as well: C becomes exactly zero without being read
    c.C[:, :, :c.n] = float("nan")
    assert _raw(c, A=0, B=0, alpha=0.0, beta=0.0) == mpg.OK
    assert np.all(c.result()[0] == 0.0)


def test_empty_problems_leave_c_untouched():
    mpg.build()
    c = Case(33, 17, 9, mpg.TF32, pad=(0, 0, 2))
    for kw in (dict(m=0), dict(n=0), dict(batch=0)):
        assert _raw(c, **kw) == mpg.OK
    assert np.array_equal(c.result()[0], c.c0[0])


@pytest.mark.parametrize("mode", MODES)
def test_single_element(mode):
    mpg.build()
    c = Case(1, 1, 1, mode, alpha=3.0, beta=0.5)
    c.run()
    eR, eQ = c.errors()
    if mode == mpg.TF32:
        assert eR <= TOL["tf32"]
    elif mode == mpg.FP32_FFMA:
        assert eR <= TOL["q16"]
    else:
        assert eQ <= TOL["q16"]


@pytest.mark.parametrize("mode", [mpg.BF16_F32ACC, mpg.TF32, mpg.SPLIT_FP16_3CHAIN])
def test_batch_strides_not_packed(mode):
    """Batches placed with gaps between them (strides larger than one matrix)."""
    import torch
    mpg.build()
    batch, m, n, k = 3, 150, 90, 70
    dt = "bf16" if mode == mpg.BF16_F32ACC else "f32"
    base = Case(m, n, k, mode, batch=batch, in_dtype=dt, b_layout=mpg.COL_MAJOR, dist="normal")
    tdt = base.A.dtype
    gapA, gapB, gapC = 1024, 512, 256
    sA = m * base.lda + gapA
    sB = n * base.ldb + gapB
    sC = m * base.ldc + gapC
    A = torch.zeros(batch * sA, dtype=tdt, device="cuda")
    B = torch.zeros(batch * sB, dtype=tdt, device="cuda")
    C = torch.full((batch * sC,), float("nan"), dtype=torch.float32, device="cuda")
    for b in range(batch):
        A[b * sA:b * sA + m * base.lda] = base.A[b].reshape(-1)
        B[b * sB:b * sB + n * base.ldb] = base.B[b].reshape(-1)
        C[b * sC:b * sC + m * base.ldc] = base.C[b].reshape(-1)
    code = mpg.BF16 if dt == "bf16" else mpg.F32
    mpg.gemm_raw(m, n, k, batch, A.data_ptr(), base.lda, sA, code, mpg.ROW_MAJOR, B.data_ptr(), base.ldb, sB,
                 code, mpg.COL_MAJOR, C.data_ptr(), base.ldc, sC, 1.0, 0.5, mode)
    torch.cuda.synchronize()
    Ch = C.cpu().numpy()
    q = {mpg.BF16_F32ACC: oracle.Q_BF16, mpg.TF32: oracle.Q_NONE,
         mpg.SPLIT_FP16_3CHAIN: oracle.Q_NONE}[mode]
    tol = {mpg.BF16_F32ACC: TOL["q16"], mpg.TF32: TOL["tf32"], mpg.SPLIT_FP16_3CHAIN: TOL["split"]}[mode]
    for b in range(batch):
        got = Ch[b * sC:b * sC + m * base.ldc].reshape(m, base.ldc)
        assert np.all(np.isnan(got[:, n:])), "padding written"
        gap = Ch[b * sC + m * base.ldc:(b + 1) * sC]
        assert np.all(np.isnan(gap)), "gap between batches written"
        ref, den = oracle.gemm(base.a[b], base.b[b], base.c0[b], 1.0, 0.5, q, q)
        assert oracle.max_rel_err(got[:, :n], ref, den) <= tol


def test_taller_than_one_grid_of_tile_rows():
    """m above 65535 tile rows of 128 (the grid's y limit): the FFMA
    comparator launches its tile rows in slices, the tensor-core paths take
    their tiles persistently.  Rows at the start, at the slice boundaries
    and at the end are checked (FFMA bit for bit against the fmaf chain)."""
    import numpy as np
    import torch
    import oracle
    import synthetic
    mpg.build()
    m, n, k = 65535 * 128 + 300, 6, 5
    a = synthetic.normal((m, k), 7001)
    b = synthetic.normal((k, n), 7002)
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    rows = np.array([0, 1, 127, 65535 * 128 - 1, 65535 * 128, 65535 * 128 + 1, m - 2, m - 1])
    for mode in (mpg.FP32_FFMA, mpg.TF32):
        C = torch.zeros((m, n), dtype=torch.float32, device="cuda")
        mpg.gemm(A, B, C, alpha=1.5, beta=0.0, mode=mode)
        torch.cuda.synchronize()
        assert mpg.device_status() == mpg.OK
        got = C[torch.from_numpy(rows).cuda()].cpu().numpy()
        if mode == mpg.FP32_FFMA:
            ref = oracle.gemm_fma_chain_f32(a[rows], b, None, 1.5, 0.0)
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        else:
            ref, den = oracle.gemm(a[rows], b, None, 1.5, 0.0)
            assert oracle.max_rel_err(got, ref, den) <= 2e-3
        del C


def test_tf32_column_major_a_too_long_for_the_transposing_copy():
    """tf32 wants A row-major: a column-major A is normally copied transposed
    into the workspace, on a grid of 32 x 32 blocks.  With k above 65535 x 32
    that grid cannot cover A's rows, and the product runs on generic loads
    instead of failing."""
    import numpy as np
    import torch
    import oracle
    mpg.build()
    m, n, k = 64, 8, 65535 * 32 + 100
    g = np.random.Generator(np.random.PCG64(7003))
    at = g.standard_normal((k, m), dtype=np.float32)        # column-major A: k lines of m
    b = g.standard_normal((k, n), dtype=np.float32)
    At, B = torch.from_numpy(at).cuda(), torch.from_numpy(b).cuda()
    C = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    ws_bytes = mpg.workspace_size_ex(m, n, k, 1, At.data_ptr(), m, 0, mpg.F32, mpg.COL_MAJOR, B.data_ptr(), n, 0,
                                     mpg.F32, mpg.ROW_MAJOR, mpg.TF32)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    mpg.gemm_raw(m, n, k, 1, At.data_ptr(), m, 0, mpg.F32, mpg.COL_MAJOR, B.data_ptr(), n, 0, mpg.F32, mpg.ROW_MAJOR,
                 C.data_ptr(), n, 0, 1.0, 0.0, mpg.TF32, ws.data_ptr(), ws_bytes, 0)
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    rows = np.repeat(np.arange(0, m, 9), n)
    cols = np.tile(np.arange(n), len(rows) // n)
    ref, den = oracle.gemm_points(at, b, k, rows, cols, a_col_major=True)
    got = C.cpu().numpy()[rows, cols]
    assert oracle.max_rel_err(got, ref, den) <= 2e-3
