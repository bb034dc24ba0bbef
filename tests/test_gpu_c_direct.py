"""GPU: the direct TMA -> tcgen05 path (fp16 / bf16 via kind::f16, fp32 via
kind::tf32) against the oracle: single tiles, ragged tails in M, N and K,
both operand layouts, padded leading dimensions, alpha/beta, batches."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
from helpers import TOL, Case

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR


@pytest.mark.parametrize("dt,mode", [("bf16", mpg.BF16_F32ACC), ("f16", mpg.FP16_F32ACC)])
@pytest.mark.parametrize("m,n,k,al,bl,pad,tile_n", [
    (128, 256, 64, R, Cm, (0, 0, 0), 0),       # one tile, both operands K-major
    (128, 256, 64, R, R, (0, 0, 0), 0),        # B N-major
    (128, 256, 64, Cm, Cm, (0, 0, 0), 0),      # A M-major
    (128, 256, 64, Cm, R, (0, 0, 0), 0),
    (300, 520, 200, R, R, (8, 8, 8), 0),       # ragged M, N, K; padded leading dims
    (257, 130, 136, Cm, Cm, (16, 24, 3), 0),
    (200, 200, 72, R, R, (0, 0, 0), 128),      # 128- and 64-wide tiles
    (200, 200, 72, R, Cm, (0, 0, 0), 64),
])
def test_direct_16bit_parity(dt, mode, m, n, k, al, bl, pad, tile_n):
    mpg.build()
    opts = mpg.options(tile_n=tile_n) if tile_n else None
    c = Case(m, n, k, mode, in_dtype=dt, a_layout=al, b_layout=bl, pad=pad, alpha=1.25, beta=-0.5,
             dist="normal", opts=opts)
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)


def test_direct_bf16_batched_and_beta_zero():
    mpg.build()
    c = Case(96, 80, 160, mpg.BF16_F32ACC, batch=5, in_dtype="bf16", a_layout=R, b_layout=Cm,
             pad=(8, 8, 4), alpha=2.0, beta=0.0, dist="normal")
    # beta == 0: C is not read, so NaN in C0 must not leak through
    c.C[:, :, :c.n] = float("nan")
    c.c0[...] = 0.0
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], eQ


@pytest.mark.parametrize("m,n,k,al,bl,pad", [
    (128, 256, 32, R, Cm, (0, 0, 0)),          # direct tf32 (both K-major)
    (310, 300, 100, R, Cm, (4, 4, 4)),
    (200, 140, 96, R, R, (0, 0, 0)),            # B N-major: generic path, K-major tiles
    (130, 70, 40, Cm, Cm, (4, 0, 0)),
])
def test_tf32_parity(m, n, k, al, bl, pad):
    mpg.build()
    c = Case(m, n, k, mpg.TF32, a_layout=al, b_layout=bl, pad=pad, alpha=1.0, beta=0.25)
    c.run()
    eR, _ = c.errors()
    assert eR <= TOL["tf32"], eR


def test_tf32_operand_rounding_model(orc, capsys):
    """Which conversion the tensor core applies to fp32 operands of
    kind::tf32: inputs whose low 13 fraction bits cover the halfway and
    above-halfway cases, multiplied by exact ones, give the rounded operand."""
    mpg.build()
    m, n, k = 128, 64, 8
    base = 1.0 + np.arange(m) / 64.0
    low = np.array([0x0FFF, 0x1000, 0x1001, 0x1FFF, 0x0001, 0x1800, 0x0800, 0x17FF], dtype=np.uint32)
    bits = (base.astype(np.float32).view(np.uint32) & ~np.uint32(0x1FFF)) | low[np.arange(m) % 8]
    col = bits.view(np.float32)
    a = np.zeros((m, k), np.float32)
    a[:, 0] = col
    b = np.zeros((k, n), np.float32)
    b[0, :] = 1.0
    c = Case(m, n, k, mpg.TF32, a_layout=R, b_layout=Cm, a=a, b=b, c0=np.zeros((m, n), np.float32))
    c.run()
    got = c.result()[0][:, 0].astype(np.float64)
    models = {
        "trunc": np.array([orc.quantize(np.array([[v]], np.float64), orc.Q_TF32_TRUNC)[0][0, 0] for v in col]),
        "rna": np.array([orc.quantize(np.array([[v]], np.float64), orc.Q_TF32_RNA)[0][0, 0] for v in col]),
        "rne": np.array([orc.quantize(np.array([[v]], np.float64), orc.Q_TF32_RNE)[0][0, 0] for v in col]),
        "none": col.astype(np.float64),
    }
    match = [name for name, v in models.items() if np.array_equal(v, got)]
    with capsys.disabled():
        print(f"\n[tf32 operand model] matches: {match}")
    assert match, "the tf32 result matches none of the rounding models"


def _round_rz(x64):
    """binary64 -> fp32 rounded toward zero."""
    f = x64.astype(np.float32)
    up = np.abs(f.astype(np.float64)) > np.abs(x64)
    f[up] = np.nextafter(f[up], np.float32(0))
    return f


def test_accumulator_rounding_model(capsys):
    """How the tensor core rounds its fp32 accumulator between MMA
    instructions.  The first instruction loads 2^20-sized values, every later
    one adds 16*c_j with c_j = 1 + j/1024, whose fraction is below the
    accumulator's ulp (1/8): round-to-nearest and truncation then part ways.
    The result is compared with both models, each applied once per
    instruction (16 products summed exactly, then rounded into fp32)."""
    mpg.build()
    m, n, steps = 128, 64, 64
    k = 16 * steps
    a = np.ones((m, k), np.float32)
    cj = (1.0 + np.arange(n) / 1024.0).astype(np.float32)
    b = np.tile(cj, (k, 1)).astype(np.float32)
    b[:16, :] = 65504.0
    c = Case(m, n, k, mpg.FP16_F32ACC, in_dtype="f16", a_layout=R, b_layout=Cm, a=a, b=b,
             c0=np.zeros((m, n), np.float32))
    c.run()
    got = c.result()[0][0].astype(np.float64)
    assert np.all(c.result()[0] == got.astype(np.float32))   # every row the same
    first = 16.0 * 65504.0
    s = 16.0 * cj.astype(np.float64)
    d_rn = np.full(n, first, np.float32)
    d_rz = np.full(n, first, np.float32)
    for _ in range(steps - 1):
        d_rn = (d_rn.astype(np.float64) + s).astype(np.float32)
        d_rz = _round_rz(d_rz.astype(np.float64) + s)
    exact = first + (steps - 1) * s
    match = [name for name, d in (("round-to-nearest", d_rn), ("truncation", d_rz))
             if np.array_equal(d.astype(np.float64), got)]
    with capsys.disabled():
        print(f"\n[fp32 accumulator model] matches: {match}; max |got-exact| = "
              f"{np.max(np.abs(got - exact)):.4g}, rn {np.max(np.abs(d_rn - exact)):.4g}, "
              f"rz {np.max(np.abs(d_rz - exact)):.4g}")
    # both models bound the error by one ulp per instruction
    assert np.max(np.abs(got - exact)) <= (steps - 1) * 0.125


@pytest.mark.parametrize("mode,dt", [(mpg.BF16_F32ACC, "bf16"), (mpg.TF32, "f32"), (mpg.SPLIT_FP16_3CHAIN, "f32")])
def test_backward_operand_roles_by_layout(mode, dt):
    """The two products of a backward pass, dA = dC . B^T and dB = A^T . dC,
    read the forward pass's row-major A (m x k) and B (k x n) buffers in place:
    B^T is B's storage read column-major (ld n), A^T is A's storage read
    column-major (ld k).  No transposed copies."""
    import torch
    mpg.build()
    m, n, k = 200, 136, 168
    import synthetic
    from helpers import round_to
    a = round_to(synthetic.normal((m, k), 91), dt)
    b = round_to(synthetic.normal((k, n), 92), dt)
    dc = round_to(synthetic.normal((m, n), 93), dt)
    td = {"bf16": torch.bfloat16, "f32": torch.float32}[dt]
    code = {"bf16": mpg.BF16, "f32": mpg.F32}[dt]
    A = torch.from_numpy(a).cuda().to(td)
    B = torch.from_numpy(b).cuda().to(td)
    dC = torch.from_numpy(dc).cuda().to(td)
    dA = torch.zeros((m, k), device="cuda")
    dB = torch.zeros((k, n), device="cuda")
    # dA (m x k) = dC (m x n, row-major ld n) . B^T (n x k: B's storage, column-major ld n)
    mpg.gemm_raw(m, k, n, 1, dC.data_ptr(), n, 0, code, R, B.data_ptr(), n, 0, code, Cm,
                 dA.data_ptr(), k, 0, 1.0, 0.0, mode)
    # dB (k x n) = A^T (k x m: A's storage, column-major ld k) . dC (m x n, row-major ld n)
    mpg.gemm_raw(k, n, m, 1, A.data_ptr(), k, 0, code, Cm, dC.data_ptr(), n, 0, code, R,
                 dB.data_ptr(), n, 0, 1.0, 0.0, mode)
    torch.cuda.synchronize()
    q = {mpg.BF16_F32ACC: oracle.Q_BF16, mpg.TF32: oracle.Q_NONE, mpg.SPLIT_FP16_3CHAIN: oracle.Q_NONE}[mode]
    tol = {mpg.BF16_F32ACC: TOL["q16"], mpg.TF32: TOL["tf32"], mpg.SPLIT_FP16_3CHAIN: TOL["split"]}[mode]
    ref, den = oracle.gemm(dc, b.T.copy(), None, 1.0, 0.0, q, q)
    assert oracle.max_rel_err(dA.cpu().numpy(), ref, den) <= tol
    ref, den = oracle.gemm(a.T.copy(), dc, None, 1.0, 0.0, q, q)
    assert oracle.max_rel_err(dB.cpu().numpy(), ref, den) <= tol
