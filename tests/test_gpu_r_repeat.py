"""GPU: the pipelines' hand-offs under repetition.  Every path is
deterministic (fixed k order, fixed chain sums), so the same product run
again must give the same bits; a buffer handed back before its readers are
done (a staging slot refilled under loads still in flight, an operand stage
overwritten before the tensor core read it) shows up as a run that differs.
Each case runs the product a dozen times on operands larger than one wave
of tiles and compares every run bit for bit with the first, which is also
checked against the oracle on sampled elements."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR

CASES = [
    # name, mode, m, n, k, b layout, options, quantisation of the sampled check
    ("s_shared_onload", mpg.SPLIT_FP16_3CHAIN, 2048, 4096, 128, Cm, dict(prepass=-1, split_lo_shared=1),
     oracle.Q_SPLIT3),
    ("s_three_onload", mpg.SPLIT_FP16_3CHAIN, 2048, 4096, 128, Cm, dict(prepass=-1), oracle.Q_SPLIT3),
    ("fp16_onload", mpg.FP16_F32ACC, 2048, 2048, 1024, R, dict(prepass=-1), oracle.Q_FP16),
    ("split3_onload_chunks", mpg.SPLIT_FP16_3CHAIN, 1024, 1024, 2048, R, dict(prepass=-1), oracle.Q_SPLIT3),
    ("split3_pass", mpg.SPLIT_FP16_3CHAIN, 1024, 1024, 2048, R, dict(prepass=1), oracle.Q_SPLIT3),
    ("generic_split1", mpg.SPLIT_FP16_1CHAIN, 640, 640, 512, R, dict(force_generic_load=1), oracle.Q_SPLIT1),
    ("bf16_pair", mpg.BF16_F32ACC, 2048, 2048, 1024, R, dict(cta_pair=1), oracle.Q_BF16),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c[0])
def test_repeated_runs_give_identical_bits(case):
    import torch
    name, mode, m, n, k, bl, kw, q = case
    mpg.build()
    a = synthetic.normal((m, k), 9100)
    b = synthetic.normal((k, n), 9200)
    if mode == mpg.BF16_F32ACC:
        A = torch.from_numpy(a).cuda().to(torch.bfloat16)
        B = torch.from_numpy(b).cuda().to(torch.bfloat16)
        a = A.float().cpu().numpy()
        b = B.float().cpu().numpy()
    else:
        A = torch.from_numpy(a).cuda()
        B = torch.from_numpy(np.ascontiguousarray(b.T) if bl == Cm else b).cuda()
    dt = mpg.BF16 if mode == mpg.BF16_F32ACC else mpg.F32
    ldb = k if bl == Cm else n
    opts = mpg.options(**kw)
    ws_bytes = mpg.workspace_size(m, n, k, 1, mode, opts)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(12):
        C = torch.empty((m, n), dtype=torch.float32, device="cuda")
        mpg.gemm_raw(m, n, k, 1, A.data_ptr(), k, 0, dt, R, B.data_ptr(), ldb, 0, dt, bl, C.data_ptr(), n, 0,
                     1.0, 0.0, mode, ws.data_ptr(), ws_bytes, 0, opts)
        outs.append(C)
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    first = outs[0].view(torch.int32)
    for i, C in enumerate(outs[1:], 1):
        diff = int((C.view(torch.int32) != first).sum().item())
        assert diff == 0, (name, i, diff)
    rows = np.random.Generator(np.random.PCG64(9300)).integers(0, m, size=400)
    cols = np.random.Generator(np.random.PCG64(9301)).integers(0, n, size=400)
    got = outs[0].cpu().numpy()[rows, cols]
    ref, den = oracle.gemm_points(a, b, k, rows, cols, a_q=q, b_q=q)
    assert oracle.max_rel_err(got, ref, den) <= 1e-5, name


@pytest.mark.parametrize("amode", ["two", "one"])
def test_fused_attention_repeated_runs_give_identical_bits(amode):
    """The fused attention's hand-offs (S read out while the next S goes in,
    the flag exchange, the P writes, the folds, the merge of key ranges)
    under repetition: a dozen runs, identical bits, and the first run within
    the bar against the oracle on sampled rows."""
    import torch
    mpg.build()
    lq, lk, d = 2048, 8192 + 77, 128
    q = synthetic.normal((lq, d), 9400)
    kk = synthetic.normal((lk, d), 9401).astype(np.float16)
    vv = synthetic.normal((lk, d), 9402).astype(np.float16)
    Q = torch.from_numpy(q).cuda()
    K, V = torch.from_numpy(kk).cuda(), torch.from_numpy(vv).cuda()
    mode = mpg.ATTN_SPLIT_2CHAIN if amode == "two" else mpg.ATTN_SPLIT_1CHAIN
    outs = [mpg.attention(Q, K, V, scale=0.125, mode=mode) for _ in range(12)]
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    first = outs[0].view(torch.int32)
    for i, O in enumerate(outs[1:], 1):
        assert int((O.view(torch.int32) != first).sum().item()) == 0, (amode, i)
    rows = np.arange(0, lq, 97)
    ref, den = oracle.attention(q[rows], kk, vv, 0.125)
    err = float(np.max(np.abs(outs[0].cpu().numpy()[rows] - ref) / den))
    assert err <= 5e-6, err
