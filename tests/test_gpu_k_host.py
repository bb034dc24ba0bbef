"""GPU parity of mpg_gemm_host: A, B and C in host memory (page-locked or
pageable), copied in, multiplied and copied back by one call, with row
chunks pipelined against the product (batches of matrices when batch > 1).
Every case is checked against the oracle, and C's padding columns in host
memory must keep their sentinel."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic
from helpers import MODE_Q, SENTINEL_BITS, TOL, round_to, sample_points

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR
NP16 = {"f32": np.float32, "f16": np.float16}


def _host(shape, dtype, pinned):
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return torch.empty(shape, dtype=tdt, pin_memory=pinned)


def _store(t, values_f32, layout_rows, dtype):
    """Write logical values into host tensor t (already shaped as stored)."""
    import torch
    t.copy_(torch.from_numpy(np.ascontiguousarray(values_f32)).to(t.dtype))


def run_host(a, b, c0, mode, dt="bf16", cdt="f32", al=R, bl=R, pad=(0, 0, 0), alpha=1.0, beta=0.0,
             pinned=True, c_stride_pad=0, opts=None):
    """a: (batch, m, k), b: (batch, k, n), c0: (batch, m, n) logical fp32 values."""
    import torch
    batch, m, k = a.shape
    n = b.shape[2]
    lda = (k if al == R else m) + pad[0]
    ldb = (n if bl == R else k) + pad[1]
    ldc = n + pad[2]
    a_outer, b_outer = (m if al == R else k), (k if bl == R else n)
    sA, sB = a_outer * lda, b_outer * ldb
    sC = m * ldc + c_stride_pad
    hA = _host((batch, sA), dt, pinned)
    hB = _host((batch, sB), dt, pinned)
    hC = _host((batch, sC), cdt, pinned)
    hA.zero_(); hB.zero_()
    Av = hA[:, :a_outer * lda].view(batch, a_outer, lda)
    Bv = hB[:, :b_outer * ldb].view(batch, b_outer, ldb)
    Av[:, :, :(k if al == R else m)] = torch.from_numpy(a if al == R else np.transpose(a, (0, 2, 1)).copy()).to(hA.dtype)
    Bv[:, :, :(n if bl == R else k)] = torch.from_numpy(b if bl == R else np.transpose(b, (0, 2, 1)).copy()).to(hB.dtype)
    # C: sentinel everywhere (padding columns and the gaps between matrices), c0 in the n columns
    if cdt == "f32":
        hC.view(torch.int32).fill_(int(np.int32(SENTINEL_BITS.view(np.int32))))
    else:
        hC.view(torch.int16).fill_(0x7E55)
    Cv = hC[:, :m * ldc].view(batch, m, ldc)
    Cv[:, :, :n] = torch.from_numpy(c0).to(hC.dtype)
    code = {"f32": mpg.F32, "f16": mpg.F16, "bf16": mpg.BF16}
    o = opts if opts is not None else mpg.options()
    o.c_dtype = code[cdt]
    ws_bytes = mpg.host_workspace_size(m, n, k, batch, lda, sA if batch > 1 else 0, code[dt], al, ldb,
                                       sB if batch > 1 else 0, code[dt], bl, ldc, sC if batch > 1 else 0,
                                       alpha, beta, mode, o)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    before = hC.clone()
    mpg.gemm_host_raw(m, n, k, batch, hA.data_ptr(), lda, sA if batch > 1 else 0, code[dt], al,
                      hB.data_ptr(), ldb, sB if batch > 1 else 0, code[dt], bl,
                      hC.data_ptr(), ldc, sC if batch > 1 else 0, alpha, beta, mode,
                      ws.data_ptr(), ws_bytes, stream.cuda_stream, o)
    stream.synchronize()
    assert mpg.device_status() == mpg.OK
    # nothing outside the n columns of each row was written
    mask = torch.ones_like(hC, dtype=torch.bool)
    mask[:, :m * ldc].view(batch, m, ldc)[:, :, :n] = False
    bits = torch.int32 if cdt == "f32" else torch.int16   # the sentinel is a NaN pattern: compare bits
    assert torch.equal(hC.view(bits)[mask], before.view(bits)[mask]), "padding of host C was written"
    return Cv[:, :, :n].float().numpy().astype(np.float64)


def _check(got, a, b, c0, q, alpha, beta, tol, cdt="f32"):
    for bi in range(a.shape[0]):
        ref, den = oracle.gemm(a[bi], b[bi], c0[bi], alpha, beta, q, q)
        if cdt == "f32":
            assert oracle.max_rel_err(got[bi], ref, den) <= tol
        else:
            ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))) - 10)
            assert np.all(np.abs(got[bi] - ref) <= ulp + tol * den)


@pytest.mark.parametrize("al,bl", [(R, R), (Cm, Cm), (R, Cm)])
def test_host_single_chunk_layouts(al, bl):
    mpg.build()
    a = round_to(synthetic.normal((1, 300, 200), 131), "bf16")
    b = round_to(synthetic.normal((1, 200, 260), 132), "bf16")
    c0 = synthetic.normal((1, 300, 260), 133)
    got = run_host(a, b, c0, mpg.BF16_F32ACC, al=al, bl=bl, pad=(8, 8, 5), alpha=1.25, beta=-0.5)
    _check(got, a, b, c0, oracle.Q_BF16, 1.25, -0.5, TOL["q16"])


@pytest.mark.parametrize("al", [R, Cm])
def test_host_row_chunks_pipelined(al, capsys):
    """8192 x 4096 x 1024 bf16 with beta: over 128 MB of inputs, so the call
    cuts A and C into row chunks; checked on sampled elements and on whole
    rows at the chunk boundaries."""
    mpg.build()
    m, n, k = 8192, 4096, 1024
    a = round_to(synthetic.normal((1, m, k), 141), "bf16")
    b = round_to(synthetic.normal((1, k, n), 142), "bf16")
    c0 = synthetic.normal((1, m, n), 143)
    got = run_host(a, b, c0, mpg.BF16_F32ACC, al=al, pad=(0, 0, 4), beta=0.5)
    rows, cols = sample_points(m, n, 2000, 144)
    ref, den = oracle.gemm_points(a[0], b[0], k, rows, cols, c0[0], 1.0, 0.5, oracle.Q_BF16, oracle.Q_BF16)
    assert oracle.max_rel_err(got[0][rows, cols], ref, den) <= TOL["q16"]
    edge = np.array([0, 4095, 4096, 8191])
    ref, den = oracle.gemm(a[0][edge], b[0], c0[0][edge], 1.0, 0.5, oracle.Q_BF16, oracle.Q_BF16)
    assert oracle.max_rel_err(got[0][edge], ref, den) <= TOL["q16"]


@pytest.mark.parametrize("c_stride_pad", [0, 24])
def test_host_batched_split_mode(c_stride_pad):
    """fp32 operands in the split mode, five matrices with padded leading
    dimensions; C's matrices packed (one copy back) or spaced apart (one copy
    back per matrix)."""
    mpg.build()
    a = synthetic.normal((5, 70, 130), 151)
    b = synthetic.normal((5, 130, 90), 152)
    c0 = synthetic.normal((5, 70, 90), 153)
    got = run_host(a, b, c0, mpg.SPLIT_FP16_3CHAIN, dt="f32", bl=Cm, pad=(4, 4, 6), beta=1.0,
                   c_stride_pad=c_stride_pad)
    _check(got, a, b, c0, oracle.Q_NONE, 1.0, 1.0, TOL["split"])


def test_host_pageable_memory_and_sixteen_bit_output():
    mpg.build()
    a = synthetic.normal((1, 130, 64), 161)
    b = synthetic.normal((1, 64, 200), 162)
    c0 = round_to(synthetic.normal((1, 130, 200), 163), "f16")
    got = run_host(a, b, c0, mpg.TF32, dt="f32", cdt="f16", bl=Cm, pad=(0, 0, 8), beta=0.25, pinned=False)
    for bi in range(1):
        ref, den = oracle.gemm(a[bi], b[bi], c0[bi], 1.0, 0.25)
        ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(ref), 2.0 ** -14))) - 10)
        assert np.all(np.abs(got[bi] - ref) <= ulp + TOL["tf32"] * den)


def test_host_k_zero_scales_c():
    mpg.build()
    a = np.zeros((1, 40, 0), np.float32)
    b = np.zeros((1, 0, 50), np.float32)
    c0 = synthetic.normal((1, 40, 50), 171)
    got = run_host(a, b, c0, mpg.FP32_FFMA, dt="f32", pad=(1, 0, 3), beta=-2.0)
    assert np.array_equal(got[0], (-2.0 * c0[0].astype(np.float32)).astype(np.float64))


def test_host_odd_leading_dimensions_run_on_aligned_device_copies():
    """bf16 host operands with odd leading dimensions: the device copies are
    padded to 16-byte lines, so the product takes the TMA path (checked here
    for values; the padding of host C is checked by run_host)."""
    mpg.build()
    a = round_to(synthetic.normal((1, 520, 301), 181), "bf16")
    b = round_to(synthetic.normal((1, 301, 263), 182), "bf16")
    c0 = synthetic.normal((1, 520, 263), 183)
    got = run_host(a, b, c0, mpg.BF16_F32ACC, al=R, bl=Cm, pad=(0, 0, 1), alpha=1.0, beta=0.5)
    _check(got, a, b, c0, oracle.Q_BF16, 1.0, 0.5, TOL["q16"])


def test_torch_gemm_host_on_cpu_tensors():
    import torch
    mpg.build()
    a = round_to(synthetic.normal((300, 200), 191), "bf16")
    b = round_to(synthetic.normal((200, 260), 192), "bf16")
    c0 = synthetic.normal((300, 260), 193)
    A = torch.from_numpy(a).to(torch.bfloat16).pin_memory()
    B = torch.from_numpy(b).to(torch.bfloat16).t().contiguous().t()     # column-major view
    C = torch.from_numpy(c0.copy())
    out = mpg.gemm_host(A, B, C, alpha=1.0, beta=0.5, mode="bf16")
    assert out is C and not C.is_cuda
    ref, den = oracle.gemm(a, b, c0, 1.0, 0.5, oracle.Q_BF16, oracle.Q_BF16)
    assert oracle.max_rel_err(C.numpy(), ref, den) <= TOL["q16"]


def test_host_full_size_bf16_8192_beta(capsys):
    """The end-to-end configuration of the benchmark: 8192^3 bf16 with beta =
    0.5 from page-locked host buffers through mpg_gemm_host (row chunks
    pipelined against the product); sampled elements and whole rows at chunk
    boundaries against the oracle."""
    mpg.build()
    n = 8192
    a = round_to(synthetic.normal((1, n, n), synthetic.SEED_A), "bf16")
    b = round_to(synthetic.normal((1, n, n), synthetic.SEED_B), "bf16")
    c0 = synthetic.normal((1, n, n), synthetic.SEED_C0)
    got = run_host(a, b, c0, mpg.BF16_F32ACC, beta=0.5)
    rows, cols = sample_points(n, n, 2000, 195)
    ref, den = oracle.gemm_points(a[0], b[0], n, rows, cols, c0[0], 1.0, 0.5, oracle.Q_BF16, oracle.Q_BF16)
    err = oracle.max_rel_err(got[0][rows, cols], ref, den)
    edge = np.array([0, 1535, 1536, 4607, 4608, 8191])
    refr, denr = oracle.gemm(a[0][edge], b[0], c0[0][edge], 1.0, 0.5, oracle.Q_BF16, oracle.Q_BF16)
    err_rows = oracle.max_rel_err(got[0][edge], refr, denr)
    with capsys.disabled():
        print(f"\n[host 8192^3 bf16: sampled {err:.3e}, rows {err_rows:.3e}]")
    assert err <= TOL["q16"] and err_rows <= TOL["q16"]
