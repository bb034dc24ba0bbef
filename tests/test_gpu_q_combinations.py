"""GPU: options and entry points in combinations the per-feature files leave
out.  The shared lo accumulator (hi*lo and lo*hi in one TMEM chain, "split
FP32 into FP16 hi + lo ..." with the lo products summed before they meet the
hi*hi chain) with batches, beta, split-K, the conversion pass and generic
loads; the TMA-store epilogue into a batched C whose matrices are separated
by gaps; and the host-memory entry with the conversion pass.  Every result is
checked against the oracle on the quantised-input problem, or bit for bit
against the same product on a path whose own parity is tested elsewhere."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import oracle
import synthetic
from helpers import SENTINEL_BITS, TOL, Case

pytestmark = pytest.mark.gpu

R, Cm = mpg.ROW_MAJOR, mpg.COL_MAJOR

SHARED = [
    # m, n, k, batch, a_layout, alpha, beta, options
    (333, 141, 777, 3, Cm, 0.75, 0.5, dict(prepass=-1, split_chunk_k=-1)),
    (256, 128, 4096, 1, R, 1.0, -1.0, dict(prepass=-1, split_chunk_k=-1, splitk=3)),
    (300, 200, 480, 2, R, -2.0, 0.25, dict(prepass=1)),
    (129, 65, 300, 2, Cm, 1.5, 1.0, dict(prepass=-1, force_generic_load=1)),
    (384, 256, 2048, 1, R, 1.0, 0.0, dict(prepass=1, split_chunk_k=-1, splitk=2)),
]


@pytest.mark.parametrize("case", SHARED, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}_b{c[3]}_{sorted(c[7])}")
def test_shared_lo_accumulator_combinations(case):
    m, n, k, batch, al, alpha, beta, kw = case
    mpg.build()
    c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, batch=batch, a_layout=al, pad=(0, 0, 3), alpha=alpha, beta=beta,
             dist="normal", seed=21, opts=mpg.options(split_lo_shared=1, **kw))
    c.run()
    eR, eQ = c.errors()
    assert eQ <= TOL["q16"], (eR, eQ)
    assert eR <= TOL["split"], (eR, eQ)


def test_shared_lo_beyond_one_chunk_keeps_separate_chains():
    """With K above one accumulation chunk the shared accumulator is not
    used: the result is the separate chains' bit for bit."""
    import torch
    mpg.build()
    m, n, k = 256, 192, 1536
    outs = []
    for shared in (0, 1):
        c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, alpha=1.0, beta=0.5, dist="normal", seed=22,
                 opts=mpg.options(prepass=-1, split_lo_shared=shared, split_chunk_k=512))
        c.run()
        outs.append(c.result())
    torch.cuda.synchronize()
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def _gapped_c(batch, m, n, stride_c, c0):
    import torch
    buf = torch.empty(batch * stride_c + 8, dtype=torch.float32, device="cuda")
    buf.view(torch.int32).fill_(int(SENTINEL_BITS.view(np.int32)))
    for bi in range(batch):
        buf[bi * stride_c:bi * stride_c + m * n].copy_(torch.from_numpy(c0[bi].reshape(-1)))
    return buf


@pytest.mark.parametrize("mode,dt,kw", [(mpg.BF16_F32ACC, "bf16", {}), (mpg.TF32, "f32", {}),
                                        (mpg.SPLIT_FP16_3CHAIN, "f32", dict(prepass=-1))])
def test_tma_store_into_gapped_batches(mode, dt, kw):
    """C's matrices 16 floats apart (TMA stores: the batch stride is a whole
    number of 16-byte chunks) and 1 float apart (register stores): same bits,
    and the gaps keep their sentinel."""
    import torch
    mpg.build()
    batch, m, n, k = 3, 200, 136, 160
    a = synthetic.normal((batch, m, k), 4100)
    b = synthetic.normal((batch, k, n), 4200)
    c0 = np.zeros((batch, m, n), np.float32)
    td = {"f32": torch.float32, "bf16": torch.bfloat16}[dt]
    code = {"f32": mpg.F32, "bf16": mpg.BF16}[dt]
    A = torch.from_numpy(a).to(td).cuda()
    b_col = mode == mpg.TF32
    B = torch.from_numpy(np.ascontiguousarray(np.transpose(b, (0, 2, 1))) if b_col else b).to(td).cuda()
    ldb = k if b_col else n
    results = []
    for gap in (16, 1):
        stride_c = m * n + gap
        buf = _gapped_c(batch, m, n, stride_c, c0)
        ws_bytes = mpg.workspace_size(m, n, k, batch, mode, mpg.options(**kw))
        ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
        mpg.gemm_raw(m, n, k, batch, A.data_ptr(), k, m * k, code, R, B.data_ptr(), ldb, k * n, code,
                     Cm if b_col else R, buf.data_ptr(), n, stride_c, 0.5, 0.0, mode, ws.data_ptr(), ws_bytes, 0,
                     mpg.options(**kw))
        torch.cuda.synchronize()
        assert mpg.device_status() == mpg.OK
        out = buf.cpu().numpy()
        for bi in range(batch):
            lo, hi = bi * stride_c + m * n, (bi + 1) * stride_c
            assert np.all(out[lo:hi].view(np.uint32) == SENTINEL_BITS), ("gap written", gap, bi)
        assert np.all(out[batch * stride_c:].view(np.uint32) == SENTINEL_BITS)
        results.append(np.stack([out[bi * stride_c:bi * stride_c + m * n].reshape(m, n) for bi in range(batch)]))
    assert np.array_equal(results[0].view(np.uint32), results[1].view(np.uint32))
    # and the values are the product's
    q = {mpg.BF16_F32ACC: oracle.Q_BF16, mpg.TF32: oracle.Q_NONE, mpg.SPLIT_FP16_3CHAIN: oracle.Q_SPLIT3}[mode]
    ain = a if dt == "f32" else A.float().cpu().numpy()
    bin_ = b if dt == "f32" else torch.from_numpy(b).to(td).float().numpy()
    for bi in range(batch):
        ref, den = oracle.gemm(ain[bi], bin_[bi], None, 0.5, 0.0, q, q)
        tol = TOL["tf32"] if mode == mpg.TF32 else TOL["q16"]
        assert oracle.max_rel_err(results[0][bi], ref, den) <= tol


def test_host_entry_with_conversion_pass_matches_device_entry():
    """mpg_gemm_host with the conversion pass forced gives the device entry's
    bits for the same options (the pass, its dependent product and the
    copies in and out, all on one stream)."""
    import torch
    mpg.build()
    batch, m, n, k = 2, 384, 320, 1024
    a = synthetic.normal((batch, m, k), 4300)
    b = synthetic.normal((batch, k, n), 4400)
    c0 = synthetic.uniform((batch, m, n), 4500)
    opts = mpg.options(prepass=1, splitk=1)     # the host entry's row chunks keep the device entry's K order
    hA, hB = torch.from_numpy(a).pin_memory(), torch.from_numpy(b).pin_memory()
    hC = torch.from_numpy(c0.copy()).pin_memory()
    ws_bytes = mpg.host_workspace_size(m, n, k, batch, k, m * k, mpg.F32, R, n, k * n, mpg.F32, R, n, m * n,
                                       1.0, 0.5, mpg.SPLIT_FP16_3CHAIN, opts)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    mpg.gemm_host_raw(m, n, k, batch, hA.data_ptr(), k, m * k, mpg.F32, R, hB.data_ptr(), n, k * n, mpg.F32, R,
                      hC.data_ptr(), n, m * n, 1.0, 0.5, mpg.SPLIT_FP16_3CHAIN, ws.data_ptr(), ws_bytes,
                      stream.cuda_stream, opts)
    stream.synchronize()
    assert mpg.device_status() == mpg.OK
    c = Case(m, n, k, mpg.SPLIT_FP16_3CHAIN, batch=batch, a=a, b=b, c0=c0, alpha=1.0, beta=0.5,
             opts=mpg.options(prepass=1, splitk=1))
    c.run()
    dev = c.result()
    assert np.array_equal(hC.numpy().view(np.uint32), dev.view(np.uint32))
    eR, eQ = c.errors(dev)
    assert eQ <= TOL["q16"] and eR <= TOL["split"], (eR, eQ)
