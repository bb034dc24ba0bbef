"""GPU: the mma.sync m16n8k16 accumulator-layout probe and the bounded-wait
self test (failure detection without a GPU fault)."""
import os

import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import synthetic

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "layout_check.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if len(line) == 2:
            vals[line[0]] = float(line[1])
    return vals


def test_mma_m16n8k16_accumulator_layout_on_hardware(orc):
    import torch
    mpg.build()
    g = _golden()
    a = synthetic.asymmetric((16, 16), 61)   # exact in fp16, no two equal
    b = synthetic.asymmetric((16, 8), 62)
    d = mpg.probe_mma_m16n8k16(torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()).cpu().numpy()
    ref, _ = orc.gemm(a.astype(np.float16), b.astype(np.float16))
    placed = np.full((16, 8), np.nan)
    for lane in range(32):
        for j in range(4):
            r, c = mpg.acc_coords(lane, j)
            placed[r, c] = d[lane, j]
    mismatched = int(np.count_nonzero(placed != ref))
    worst = float(np.max(np.abs(placed - ref)))
    assert placed.size == g["points"]
    assert mismatched == g["mismatched"]
    assert worst == g["worst_abs_diff"]
    # a transposed or half-swapped map would not have matched
    swapped = placed.reshape(2, 8, 8)[::-1].reshape(16, 8)
    assert np.count_nonzero(swapped != ref) > 0


def test_bounded_wait_expires_and_reports():
    import torch
    mpg.build()
    assert mpg.device_status() == mpg.OK
    st = mpg.selftest_wait_timeout(5_000_000)      # 5 ms on a barrier nothing arrives at
    assert st == mpg.ERR_TIMEOUT
    # the context is intact: the status word was cleared and work still runs
    assert mpg.device_status() == mpg.OK
    x = torch.ones(4, device="cuda") * 2
    torch.cuda.synchronize()
    assert float(x.sum()) == 8.0
