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


@pytest.mark.parametrize("packed", [False, True])
def test_fma_rate_probe_does_its_work(packed):
    """The fp32 multiply-add throughput probe: every block's chains end at
    their exact values, and the measured rate is a plausible fraction of the
    pipe's nominal rate (SMs x 128 lanes x 2 flop x the maximum SM clock)."""
    import torch
    mpg.build()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    blocks, iters = 4 * sms, 2048
    out = mpg.probe_fma_rate(blocks, iters, packed)
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    assert torch.all(out == 496 + 32 * iters)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(5):
        mpg.probe_fma_rate(blocks, iters, packed, out=out)
    e1.record()
    torch.cuda.synchronize()
    tflops = 2.0 * 32 * iters * 256 * blocks * 5 / (e0.elapsed_time(e1) * 1e-3) / 1e12
    nominal = sms * 128 * 2 * 2.07e9 / 1e12
    assert 0.3 * nominal < tflops < 1.05 * nominal, (tflops, nominal)
