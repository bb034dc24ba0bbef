"""GPU: the epilogue's shared-memory staging, run alone by
mpg_probe_epilogue_staging with the product epilogues' own code.  Each warp
moves 32 x 32 fp32 blocks through its staging buffer (lane l writes row l;
the warp reads the block back by 16-byte chunks of rows, or by columns), so
the copy must equal the input bit for bit.  The same calls are the workload
of the staging bank-conflict profile."""
import numpy as np
import pytest

import mixed_precision_matmul_gb300 as mpg
import synthetic

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("scalar", [False, True])
@pytest.mark.parametrize("nblocks", [1, 7, 16384])
def test_staging_round_trip_is_exact(scalar, nblocks):
    import torch
    mpg.build()
    x = synthetic.asymmetric((nblocks, 32, 32), 171 + nblocks)
    bits = x.view(np.uint32).copy()
    # a few special values: signed zero, infinities, a NaN payload, subnormals
    bits.reshape(-1)[:6] = [0x80000000, 0x7F800000, 0xFF800000, 0x7FC0DEAD, 0x00000001, 0x807FFFFF]
    xin = torch.from_numpy(bits.view(np.float32)).cuda()
    out = mpg.probe_epilogue_staging(xin, scalar=scalar)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32), bits)


def test_staging_probe_rejects_bad_arguments():
    import torch
    mpg.build()
    x = torch.zeros(2048, dtype=torch.float32, device="cuda")
    L = mpg.lib()
    assert L.mpg_probe_epilogue_staging(x.data_ptr() + 4, x.data_ptr(), 1, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_epilogue_staging(x.data_ptr(), x.data_ptr(), 1, 2, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_epilogue_staging(x.data_ptr(), x.data_ptr(), 0, 0, None) == mpg.OK
