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


def _run_pair(m, n, k, mode, seed, alpha, beta, opts=None, a_layout=mpg.ROW_MAJOR, expect_split=True):
    """One call of each entry on the same inputs: mpg_gemm_ex with a caller
    workspace of the scratch's size, then mpg_gemm_noalloc.  Returns both
    results."""
    import torch
    a = synthetic.uniform((m, k), 1000 + seed)
    b = synthetic.uniform((k, n), 2000 + seed)
    c0 = synthetic.uniform((m, n), 3000 + seed)
    if a_layout == mpg.ROW_MAJOR:
        A, lda = torch.from_numpy(a).cuda(), k
    else:
        A, lda = torch.from_numpy(np.ascontiguousarray(a.T)).cuda(), m
    B = torch.from_numpy(b).cuda()
    C_ref = torch.from_numpy(c0).cuda()
    C_new = torch.from_numpy(c0).cuda()
    if expect_split:   # the case really uses split-K scratch
        assert 0 < mpg.workspace_size(m, n, k, 1, mode, opts) <= SCRATCH_BYTES
    ws = torch.empty(SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    ref_opts = opts if opts is not None else mpg.options()
    ref_opts.tail_split = -1
    mpg.gemm_raw(m, n, k, 1, A.data_ptr(), lda, 0, mpg.F32, a_layout, B.data_ptr(), n, 0, mpg.F32,
                 mpg.ROW_MAJOR, C_ref.data_ptr(), n, 0, alpha, beta, mode, ws.data_ptr(), SCRATCH_BYTES, stream,
                 ref_opts)
    mpg.gemm_noalloc_raw(m, n, k, 1, A.data_ptr(), lda, 0, mpg.F32, a_layout, B.data_ptr(), n, 0,
                         mpg.F32, mpg.ROW_MAJOR, C_new.data_ptr(), n, 0, alpha, beta, mode, stream, opts)
    torch.cuda.synchronize()
    assert mpg.device_status() == mpg.OK
    return C_new.cpu().numpy(), C_ref.cpu().numpy()


def test_noalloc_matches_workspace_entry_on_consecutive_calls():
    mpg.build()
    # calls in a row sharing the static scratch, different shapes, modes
    # and split counts: a later call must not see an earlier one's partial
    # sums.  The results are the workspace entry's bit for bit.
    cases = [
        (256, 128, 8192, mpg.SPLIT_FP16_3CHAIN, 1, 1.0, 0.0, None, mpg.ROW_MAJOR, True),
        (384, 96, 4096, mpg.TF32, 2, 0.5, -1.5, mpg.options(splitk=7), mpg.ROW_MAJOR, True),
        (256, 128, 8192, mpg.SPLIT_FP16_3CHAIN, 3, 2.0, 0.25, None, mpg.ROW_MAJOR, True),
        # one split, and a column-major tf32 A, which the planner copies
        # transposed into the scratch before the product
        (300, 200, 480, mpg.TF32, 4, 1.0, 0.5, None, mpg.COL_MAJOR, False),
    ]
    for m, n, k, mode, seed, alpha, beta, opts, al, split in cases:
        got, ref = _run_pair(m, n, k, mode, seed, alpha, beta, opts, al, split)
        assert np.array_equal(got, ref), (m, n, k, mode, float(np.max(np.abs(got - ref))))


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
