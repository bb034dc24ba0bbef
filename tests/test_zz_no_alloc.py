"""GPU: mpg_gemm_noalloc, the product for callers that cannot allocate device
memory (plugins whose host framework owns all device memory, services that
forbid allocation after start-up).  It must give the same result as mpg_gemm
with a caller workspace, on consecutive calls that share its static scratch,
and reject problems whose split-K partial sums do not fit that scratch.

This file is collected last on purpose."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import synthetic

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 * 1024 * 1024


def _den(a, b, c0, alpha, beta):
    return abs(alpha) * (np.abs(a.astype(np.float64)) @ np.abs(b.astype(np.float64))) + \
        abs(beta) * np.abs(c0.astype(np.float64))


def _run_pair(m, n, k, mode, seed, alpha, beta, opts=None):
    import torch
    a = synthetic.uniform((m, k), 1000 + seed)
    b = synthetic.uniform((k, n), 2000 + seed)
    c0 = synthetic.uniform((m, n), 3000 + seed)
    A = torch.from_numpy(a).cuda()
    B = torch.from_numpy(b).cuda()
    C_ref = torch.from_numpy(c0).cuda()
    C_new = torch.from_numpy(c0).cuda()
    ws_bytes = mpg.workspace_size(m, n, k, 1, mode, opts)
    assert 0 < ws_bytes <= SCRATCH_BYTES        # the case really uses split-K scratch
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    mpg.gemm_raw(m, n, k, 1, A.data_ptr(), k, 0, mpg.F32, mpg.ROW_MAJOR, B.data_ptr(), n, 0, mpg.F32,
                 mpg.ROW_MAJOR, C_ref.data_ptr(), n, 0, alpha, beta, mode, ws.data_ptr(), ws_bytes, stream, opts)
    mpg.gemm_noalloc_raw(m, n, k, 1, A.data_ptr(), k, 0, mpg.F32, mpg.ROW_MAJOR, B.data_ptr(), n, 0,
                         mpg.F32, mpg.ROW_MAJOR, C_new.data_ptr(), n, 0, alpha, beta, mode, stream, opts)
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    got, ref = C_new.cpu().numpy().astype(np.float64), C_ref.cpu().numpy().astype(np.float64)
    return float(np.max(np.abs(got - ref) / _den(a, b, c0, alpha, beta)))


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    mpg.build()
    # two calls in a row sharing the static scratch, different shapes, modes
    # and split counts: the second must not see the first's partial sums
    e1 = _run_pair(256, 128, 8192, mpg.SPLIT_FP16_3CHAIN, 1, 1.0, 0.0)
    e2 = _run_pair(384, 96, 4096, mpg.TF32, 2, 0.5, -1.5, mpg.options(splitk=7))
    e3 = _run_pair(256, 128, 8192, mpg.SPLIT_FP16_3CHAIN, 3, 2.0, 0.25)
    assert max(e1, e2, e3) <= 1e-5, (e1, e2, e3)


def test_noalloc_rejects_partials_beyond_the_scratch():
    import torch
    mpg.build()
    m, n, k = 2048, 1024, 4096
    opts = mpg.options(splitk=4)                 # 4 x 2048 x 1024 x 4 B = 32 MiB > 16 MiB
    A = torch.zeros((m, k), device="cuda")
    B = torch.zeros((k, n), device="cuda")
    C = torch.zeros((m, n), device="cuda")
    st = mpg.gemm_noalloc_raw(m, n, k, 1, A.data_ptr(), k, 0, mpg.F32, mpg.ROW_MAJOR, B.data_ptr(), n, 0,
                              mpg.F32, mpg.ROW_MAJOR, C.data_ptr(), n, 0, 1.0, 0.0, mpg.TF32, 0, opts,
                              check=False)
    assert st == mpg.ERR_WORKSPACE
    assert "static scratch" in mpg.last_error()
