"""GPU: fp16 / bf16 output.  The fp32 result alpha*acc + beta*C (beta*C read
in 16 bits) is rounded once to the output type; checked against the oracle
within one output ulp plus the mode's error bar, on every path that writes C
(tensor-core epilogue, split-K reduction, C = beta*C for k == 0, FFMA)."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic
from helpers import MODE_Q, MODE_QB, TOL, round_to, stored

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR


def _ulp(x, out):
    a = np.maximum(np.abs(x), 2.0 ** -14 if out == "f16" else 2.0 ** -126)
    e = np.floor(np.log2(a))
    return np.exp2(e - (10 if out == "f16" else 7))


def _run(mode, dt, out, m, n, k, al=R, bl=R, beta=0.5, opts=None, ldc_pad=0):
    import torch
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}
    a = round_to(synthetic.normal((m, k), 101), dt)
    b = round_to(synthetic.normal((k, n), 102), dt)
    c0 = round_to(synthetic.normal((m, n), 103), out)
    lda, ldb = max(k if al == R else m, 1), max(n if bl == R else k, 1)
    A = torch.from_numpy(stored(a[None], al, lda)[0]).cuda().to(tdt[dt])
    B = torch.from_numpy(stored(b[None], bl, ldb)[0]).cuda().to(tdt[dt])
    ldc = n + ldc_pad
    C = torch.zeros((m, ldc), dtype=tdt[out], device="cuda")
    C[:, :n] = torch.from_numpy(c0).cuda().to(tdt[out])
    o = opts if opts is not None else mpg.options()
    o.c_dtype = {"f16": mpg.F16, "bf16": mpg.BF16}[out]
    code = {"f32": mpg.F32, "f16": mpg.F16, "bf16": mpg.BF16}[dt]
    ws_bytes = mpg.workspace_size(m, n, k, 1, mode, o)
    ws = torch.empty(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    mpg.gemm_raw(m, n, k, 1, A.data_ptr(), lda, 0, code, al, B.data_ptr(), ldb, 0, code, bl,
                 C.data_ptr(), ldc, 0, 1.25, beta, mode, ws.data_ptr(), ws_bytes, 0, o)
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    got = C[:, :n].float().cpu().numpy().astype(np.float64)
    q = MODE_Q.get(mode, oracle.Q_NONE)
    ref, den = oracle.gemm(a, b, c0, 1.25, beta, q, MODE_QB.get(mode, q))
    return got, ref, den


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("mode,dt", [(mpg.BF16_F32ACC, "bf16"), (mpg.FP16_F32ACC, "f32"), (mpg.TF32, "f32"),
                                     (mpg.SPLIT_FP16_3CHAIN, "f32"), (mpg.FP32_FFMA, "f32")])
@pytest.mark.parametrize("m,n,k,al,bl,pad", [(300, 260, 190, R, R, 0), (129, 520, 64, Cm, Cm, 4),
                                              (150, 100, 33, R, Cm, 1)])
def test_sixteen_bit_output(out, mode, dt, m, n, k, al, bl, pad):
    mpg.build()
    got, ref, den = _run(mode, dt, out, m, n, k, al, bl, ldc_pad=pad)
    tol = TOL["tf32"] if mode == mpg.TF32 else TOL["q16"]
    assert np.all(np.abs(got - ref) <= _ulp(ref, out) + tol * den)


@pytest.mark.parametrize("out", ["f16", "bf16"])
def test_sixteen_bit_output_split_k_and_scale(out):
    mpg.build()
    got, ref, den = _run(mpg.SPLIT_FP16_3CHAIN, "f32", out, 128, 128, 4096, opts=mpg.options(splitk=6))
    assert np.all(np.abs(got - ref) <= _ulp(ref, out) + TOL["split"] * den)
    got, ref, den = _run(mpg.BF16_F32ACC, "bf16", out, 70, 90, 0, beta=-0.75)   # k == 0: C = beta*C
    assert np.all(np.abs(got - ref) <= _ulp(ref, out))


def test_torch_api_output_type_follows_c():
    """gemm() takes the output type from C's dtype, also when the caller's
    options say otherwise."""
    import torch
    mpg.build()
    m, n, k = 200, 136, 96
    a = synthetic.normal((m, k), 111)
    b = synthetic.normal((k, n), 112)
    A, B = torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()
    ref, den = oracle.gemm(a, b, None, 1.0, 0.0, oracle.Q_FP16, oracle.Q_FP16)
    C16 = torch.zeros((m, n), dtype=torch.bfloat16, device="cuda")
    mpg.gemm(A, B, C16, mode="fp16")
    got = C16.float().cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - ref) <= _ulp(ref, "bf16") + TOL["q16"] * den)
    C32 = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    mpg.gemm(A, B, C32, mode="fp16", opts=mpg.options(c_dtype=mpg.F16))
    torch.cuda.synchronize()
    assert oracle.max_rel_err(C32.cpu().numpy(), ref, den) <= TOL["q16"]


@pytest.mark.parametrize("out", ["f16", "bf16"])
@pytest.mark.parametrize("name,mode,dt,m,n,k,beta,kw", [
    ("pair_tail", mpg.BF16_F32ACC, "bf16", 520, 516, 320, 0.5, dict(cta_pair=1, tail_split=1)),
    ("pair_beta0", mpg.BF16_F32ACC, "bf16", 300, 260, 190, 0.0, dict(cta_pair=1)),
    ("pass_split3", mpg.SPLIT_FP16_3CHAIN, "f32", 300, 200, 300, 0.5, dict(prepass=1)),
    ("pass_split3_shared", mpg.SPLIT_FP16_3CHAIN, "f32", 300, 200, 300, 0.0, dict(prepass=1, split_lo_shared=1)),
    ("onload_fp16_beta0", mpg.FP16_F32ACC, "f32", 257, 132, 100, 0.0, dict(prepass=-1)),
    ("generic_split4", mpg.SPLIT_FP16_4CHAIN, "f32", 140, 70, 96, 0.5, dict(force_generic_load=1)),
])
def test_sixteen_bit_output_on_other_paths(out, name, mode, dt, m, n, k, beta, kw):
    """16-bit C from the CTA pairs (with the split tail's fixup, and with
    beta = 0), the conversion pass's copies (three chains and the shared lo
    accumulator), the load-stage converter and generic loads."""
    mpg.build()
    got, ref, den = _run(mode, dt, out, m, n, k, beta=beta, opts=mpg.options(**kw))
    tol = TOL["split"] if mode in (mpg.SPLIT_FP16_3CHAIN, mpg.SPLIT_FP16_4CHAIN) else TOL["q16"]
    assert np.all(np.abs(got - ref) <= _ulp(ref, out) + tol * den), name
