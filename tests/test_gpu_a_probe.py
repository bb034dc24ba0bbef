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


def _pack_pairs(vals16):
    """(..., 2) fp16 values -> uint32 words, element 0 in the low half."""
    bits = vals16.astype(np.float16).view(np.uint16).astype(np.uint32)
    return (bits[..., 0] | (bits[..., 1] << 16)).astype(np.uint32)


def test_operand_fragment_maps_on_hardware(orc):
    """Fragments packed on the host with the A / B maps, loaded verbatim by
    one mma.sync: the product must equal the host product exactly, so a wrong
    map (transposed, half-swapped, registers exchanged) fails."""
    import torch
    mpg.build()
    a = synthetic.asymmetric((16, 16), 63)
    b = synthetic.asymmetric((16, 8), 64)
    af = np.zeros((32, 8), np.float32)
    bf = np.zeros((32, 4), np.float32)
    for lane in range(32):
        for i in range(8):
            r, c = mpg.frag_a_coords(lane, i)
            af[lane, i] = a[r, c]
        for i in range(4):
            k, n = mpg.frag_b_coords(lane, i)
            bf[lane, i] = b[k, n]
    A = torch.from_numpy(_pack_pairs(af.reshape(32, 4, 2)).view(np.int32)).cuda()
    B = torch.from_numpy(_pack_pairs(bf.reshape(32, 2, 2)).view(np.int32)).cuda()
    d = mpg.probe_mma_m16n8k16_fragments(A, B).cpu().numpy()
    ref, _ = orc.gemm(a.astype(np.float16), b.astype(np.float16))
    placed = np.full((16, 8), np.nan)
    for lane in range(32):
        for j in range(4):
            r, c = mpg.acc_coords(lane, j)
            placed[r, c] = d[lane, j]
    assert np.array_equal(placed, ref)
    # the same fragments with A's registers 1 and 2 exchanged give another product
    A2 = torch.from_numpy(_pack_pairs(af.reshape(32, 4, 2))[:, [0, 2, 1, 3]].copy().view(np.int32)).cuda()
    d2 = mpg.probe_mma_m16n8k16_fragments(A2, B).cpu().numpy()
    assert not np.array_equal(d2, d)


@pytest.mark.parametrize("n", [64, 128, 256])
def test_tmem_accumulator_map_on_hardware(orc, n):
    """One k-block (K = 64, four tcgen05.mma kind::f16) of the one-CTA path;
    the raw tcgen05.ld registers placed on the host with the exported
    mpg_tmem_acc_coords must equal the host product at every one of the
    128 x n points (integer inputs: every product and sum is exact).  A row
    map shifted by a lane or a quarter, or a transposed column order inside
    a load, would not have matched."""
    import torch
    mpg.build()
    g = np.random.Generator(np.random.PCG64(7100 + n))
    a = g.integers(-3, 4, size=(128, 64)).astype(np.float32)
    bt = g.integers(-3, 4, size=(n, 64)).astype(np.float32)     # row j = column j of B
    d = mpg.probe_tmem_acc(torch.from_numpy(a).cuda(), torch.from_numpy(bt).cuda()).cpu().numpy()
    assert mpg.device_status() == mpg.OK
    ref, _ = orc.gemm(a.astype(np.float16), np.ascontiguousarray(bt.T).astype(np.float16))
    placed = np.full((128, n), np.nan)
    for warp in range(4):
        for lane in range(32):
            for c in range(n // 32):
                for reg in range(32):
                    r, col = mpg.tmem_acc_coords(warp, lane, reg, 32 * c)
                    assert np.isnan(placed[r, col])             # no point placed twice
                    placed[r, col] = d[warp, lane, c, reg]
    assert int(np.count_nonzero(placed != ref)) == 0
    # wrong maps: lanes shifted by one, quarters swapped, columns reversed in a load
    assert np.count_nonzero(np.roll(placed, 1, axis=0) != ref) > 0
    assert np.count_nonzero(placed.reshape(4, 32, n)[[1, 0, 3, 2]].reshape(128, n) != ref) > 0
    assert np.count_nonzero(placed.reshape(128, n // 32, 32)[:, :, ::-1].reshape(128, n) != ref) > 0


@pytest.mark.parametrize("n", [64, 128, 256])
def test_tmem_accumulator_map_on_hardware_cta_pair(orc, n):
    """The M = 256 map on a CTA pair (cta_group::2): the raw registers of both
    CTAs placed with mpg_tmem_acc_coords(256, rank, ...) equal the host
    product at every one of the 256 x n points; swapping the CTAs' halves
    would not."""
    import torch
    mpg.build()
    g = np.random.Generator(np.random.PCG64(7200 + n))
    a = g.integers(-3, 4, size=(256, 64)).astype(np.float32)
    bt = g.integers(-3, 4, size=(n, 64)).astype(np.float32)
    d = mpg.probe_tmem_acc_pair(torch.from_numpy(a).cuda(), torch.from_numpy(bt).cuda()).cpu().numpy()
    assert mpg.device_status() == mpg.OK
    ref, _ = orc.gemm(a.astype(np.float16), np.ascontiguousarray(bt.T).astype(np.float16))
    placed = np.full((256, n), np.nan)
    for rank in range(2):
        for warp in range(4):
            for lane in range(32):
                for c in range(n // 32):
                    for reg in range(32):
                        r, col = mpg.tmem_acc_coords(warp, lane, reg, 32 * c, m_shape=256, cta_rank=rank)
                        assert np.isnan(placed[r, col])
                        placed[r, col] = d[rank, warp, lane, c, reg]
    assert int(np.count_nonzero(placed != ref)) == 0
    assert np.count_nonzero(np.concatenate([placed[128:], placed[:128]]) != ref) > 0
