"""CPU tests of the C ABI: the library loads and exports every declared
symbol, arguments are validated on the host before anything launches, and the
host decode of accumulator fragments satisfies the properties its page lists
(checked against the oracle's independent transcription of the PTX formulas).
"""
import ctypes

import pytest

import mixed_precision_matmul_gb300 as mpg


@pytest.fixture(scope="module")
def L():
    mpg.build()
    return mpg.lib()


def test_every_declared_symbol_is_exported(L):
    names = mpg.header_functions()
    assert len(names) >= 14
    for name in names:
        assert hasattr(L, name), f"{name} declared in mpgemm.h but not exported"


def test_version_and_options_init(L):
    assert L.mpg_version() >= 100
    o = mpg.options()
    assert (o.split_exp_a, o.split_exp_b, o.splitk, o.force_generic_load, o.tile_n, o.wait_timeout_ns,
            o.split_chunk_k, o.prepass, o.c_dtype, o.cta_pair, o.tail_split) == (0,) * 11


# ---------------------------------------------------------------- validation
def _call(m=64, n=64, k=64, batch=1, A=16, lda=64, sA=0, adt=mpg.F32, alay=mpg.ROW_MAJOR,
          B=16, ldb=64, sB=0, bdt=mpg.F32, blay=mpg.ROW_MAJOR, C=16, ldc=64, sC=0,
          alpha=1.0, beta=0.0, mode=mpg.TF32, opts=None):
    return mpg.gemm_raw(m, n, k, batch, A, lda, sA, adt, alay, B, ldb, sB, bdt, blay, C, ldc, sC,
                        alpha, beta, mode, opts=opts, check=False)


@pytest.mark.parametrize("kw,expect", [
    (dict(m=-1), mpg.ERR_INVALID_ARG),
    (dict(k=-5), mpg.ERR_INVALID_ARG),
    (dict(batch=-1), mpg.ERR_INVALID_ARG),
    (dict(m=2 ** 31), mpg.ERR_INVALID_ARG),
    (dict(lda=63), mpg.ERR_INVALID_ARG),                           # row-major A needs lda >= k
    (dict(alay=mpg.COL_MAJOR, m=100, lda=99), mpg.ERR_INVALID_ARG),  # col-major A needs lda >= m
    (dict(ldb=10), mpg.ERR_INVALID_ARG),
    (dict(blay=mpg.COL_MAJOR, k=70, lda=70, ldb=69), mpg.ERR_INVALID_ARG),
    (dict(ldc=63), mpg.ERR_INVALID_ARG),
    (dict(sA=-1), mpg.ERR_INVALID_ARG),
    (dict(batch=2, sC=64 * 63 + 63), mpg.ERR_INVALID_ARG),        # batch matrices of C overlap
    (dict(adt=mpg.F16, bdt=mpg.F16, mode=mpg.TF32), mpg.ERR_UNSUPPORTED),
    (dict(adt=mpg.BF16, bdt=mpg.BF16, mode=mpg.FP16_F32ACC), mpg.ERR_UNSUPPORTED),
    (dict(adt=mpg.F16, bdt=mpg.F16, mode=mpg.SPLIT_FP16_3CHAIN), mpg.ERR_UNSUPPORTED),
    (dict(adt=mpg.F16, bdt=mpg.F32, mode=mpg.FP16_F32ACC), mpg.ERR_UNSUPPORTED),
    (dict(mode=17), mpg.ERR_UNSUPPORTED),
    (dict(adt=7), mpg.ERR_INVALID_ARG),
    (dict(alay=3), mpg.ERR_INVALID_ARG),
    (dict(C=0), mpg.ERR_INVALID_ARG),
    (dict(A=0), mpg.ERR_INVALID_ARG),
    (dict(C=18), mpg.ERR_INVALID_ARG),                             # C not 4-byte aligned
    (dict(A=18), mpg.ERR_INVALID_ARG),                             # fp32 A not 4-byte aligned
])
def test_invalid_arguments_rejected_before_launch(L, kw, expect):
    assert _call(**kw) == expect
    assert mpg.last_error() != ""


def test_option_ranges_rejected(L):
    assert _call(opts=mpg.options(split_exp_a=101)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(splitk=-2)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(wait_timeout_ns=-1)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(cta_pair=2)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(cta_pair=-2)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(c_dtype=3)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(tail_split=2)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(tail_split=-2)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(split_plain_lo=2)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(split_plain_lo=-1)) == mpg.ERR_INVALID_ARG
    assert _call(opts=mpg.options(split_lo_shared=2)) == mpg.ERR_INVALID_ARG


def test_probe_tmem_arguments_rejected_before_launch(L):
    assert L.mpg_probe_tmem_acc(None, None, 64, None, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_tmem_acc(16, 16, 96, 16, None) == mpg.ERR_INVALID_ARG     # n not 64 / 128 / 256
    assert L.mpg_probe_tmem_acc(8, 16, 64, 16, None) == mpg.ERR_INVALID_ARG      # A not 16-byte aligned
    assert L.mpg_probe_tmem_acc(16, 16, 64, 2, None) == mpg.ERR_INVALID_ARG      # D not 4-byte aligned
    assert L.mpg_probe_tmem_acc_pair(None, None, 64, None, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_tmem_acc_pair(16, 16, 32, 16, None) == mpg.ERR_INVALID_ARG     # n not 64 / 128 / 256
    assert L.mpg_probe_tmem_acc_pair(16, 24, 64, 16, None) == mpg.ERR_INVALID_ARG     # B not 16-byte aligned


def test_fma_probe_arguments_rejected_before_launch(L):
    assert L.mpg_probe_fma_rate(None, 1, 1, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_fma_rate(2, 1, 1, 0, None) == mpg.ERR_INVALID_ARG          # out not 4-byte aligned
    assert L.mpg_probe_fma_rate(16, 0, 1, 0, None) == mpg.ERR_INVALID_ARG         # no blocks
    assert L.mpg_probe_fma_rate(16, 65536, 1, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_fma_rate(16, 1, 0, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_fma_rate(16, 1, (1 << 19) + 1, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_fma_rate(16, 1, 1, 2, None) == mpg.ERR_INVALID_ARG          # packed not 0 / 1


def test_staging_probe_arguments_rejected_before_launch(L):
    assert L.mpg_probe_epilogue_staging(None, None, -1, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_epilogue_staging(None, None, 1, 0, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_epilogue_staging(16, 32, 1, 5, None) == mpg.ERR_INVALID_ARG
    assert L.mpg_probe_epilogue_staging(None, None, 0, 0, None) == mpg.OK    # nothing to do


def test_host_entry_rejects_a_small_workspace_before_any_copy(L):
    # host-buffer product: the workspace check precedes every copy and launch
    need = mpg.host_workspace_size(64, 64, 64, 1, 64, 0, mpg.F32, mpg.ROW_MAJOR, 64, 0, mpg.F32, mpg.ROW_MAJOR,
                                   64, 0, 1.0, 0.0, mpg.TF32)
    assert need >= 3 * 64 * 64 * 4
    st = mpg.gemm_host_raw(64, 64, 64, 1, 16, 64, 0, mpg.F32, mpg.ROW_MAJOR, 16, 64, 0, mpg.F32, mpg.ROW_MAJOR,
                           16, 64, 0, 1.0, 0.0, mpg.TF32, 256, need - 256, check=False)
    assert st == mpg.ERR_WORKSPACE and "workspace" in mpg.last_error()
    st = mpg.gemm_host_raw(64, 64, 64, 1, 16, 63, 0, mpg.F32, mpg.ROW_MAJOR, 16, 64, 0, mpg.F32, mpg.ROW_MAJOR,
                           16, 64, 0, 1.0, 0.0, mpg.TF32, 256, need, check=False)
    assert st == mpg.ERR_INVALID_ARG


def test_empty_problems_are_noops_without_a_device(L):
    # m, n or batch zero: nothing to do, no device needed, NULL pointers fine
    assert _call(m=0, A=0, B=0, C=0) == mpg.OK
    assert _call(n=0, A=0, B=0, C=0) == mpg.OK
    assert _call(batch=0, A=0, B=0, C=0) == mpg.OK


def test_alpha_zero_does_not_need_operands(L):
    # alpha == 0: A and B are not read, so NULL operands pass validation
    # (the call then needs a device, which this host does not have)
    st = _call(alpha=0.0, A=0, B=0)
    assert st in (mpg.OK, mpg.ERR_NO_DEVICE)


def _align256(x):
    return (x + 255) // 256 * 256


def _tail_bytes(tiles):
    # two halves of fp32 partial sums per 256 x 256 tile, one counter per
    # epilogue warp piece (16 per tile)
    return _align256(tiles * 2 * 256 * 256 * 4) + _align256(tiles * 16 * 4)


SMS = 152   # the queries' SM count without a device


def _pad8(x):
    return (x + 7) // 8 * 8


def _copy_room(m, n, k, es, batch=1):
    # aligned copies of A and B at the larger of the two line paddings
    return (_align256(batch * max(m * _pad8(k), k * _pad8(m)) * es) +
            _align256(batch * max(k * _pad8(n), n * _pad8(k)) * es))


def test_workspace_size_of_small_and_ffma_problems_is_zero(L):
    assert mpg.workspace_size(0, 8, 8, 1, mpg.TF32) == 0
    assert mpg.workspace_size(64, 64, 64, 1, mpg.FP32_FFMA) == 0
    assert mpg.workspace_size(256, 256, 256, 1, mpg.BF16_F32ACC) == 0     # below 2^32 multiply-adds
    assert mpg.workspace_size(128, 16384, 4096, 1, mpg.TF32) == 0         # m < 256 (and no split-K)


def test_sizes_only_query_reserves_aligned_copies_for_large_products(L):
    # the sizes-only query cannot see leading dimensions: large 16-bit and
    # tf32 products get room for aligned copies of both operands, which the
    # exact query leaves out for aligned operands
    never = mpg.options(tail_split=-1)
    n = 8192
    assert mpg.workspace_size(n, n, n, 1, mpg.BF16_F32ACC, never) == _copy_room(n, n, n, 2)
    assert mpg.workspace_size(n, n, n, 1, mpg.TF32) == _copy_room(n, n, n, 4)
    m, n2, k = 8191, 8177, 8183
    assert mpg.workspace_size(m, n2, k, 1, mpg.BF16_F32ACC, never) == _copy_room(m, n2, k, 2)
    assert mpg.workspace_size(m, n2, k, 1, mpg.BF16_F32ACC, mpg.options(tail_split=-1, prepass=-1)) == 0
    assert mpg.workspace_size(m, n2, k, 1, mpg.BF16_F32ACC, mpg.options(tail_split=-1,
                                                                        force_generic_load=1)) == 0
    aligned = mpg.workspace_size_ex(n, n, n, 1, 256, n, 0, mpg.BF16, mpg.ROW_MAJOR, 256, n, 0, mpg.BF16,
                                    mpg.ROW_MAJOR, mpg.BF16_F32ACC, never)
    assert aligned == 0


def test_workspace_holds_the_split_tail(L):
    # fp16 / bf16 products with 1 to 6 full rounds of 256 x 256 tiles on
    # SMs / 2 clusters and k >= 8192: up to SMs / 4 tiles cut in two, after
    # the aligned-copy room of the sizes-only query
    q = _tail_bytes(SMS // 4)

    def ws(m, n, k, mode, **kw):
        return mpg.workspace_size(m, n, k, 1, mode, mpg.options(**kw) if kw else None)

    def room(m, n, k, mode):
        return _copy_room(m, n, k, 4 if mode == mpg.TF32 else 2)

    for m, n, k, mode, tail in ((2560, 2560, 8192, mpg.BF16_F32ACC, True),   # 100 tiles
                                (4096, 4096, 8192, mpg.FP16_F32ACC, True),   # 256 tiles
                                (4096, 4096, 8191, mpg.FP16_F32ACC, True),   # 128 k-blocks
                                (4096, 4096, 8128, mpg.FP16_F32ACC, False),  # 127 k-blocks
                                (8192, 8192, 8192, mpg.BF16_F32ACC, False),  # 13 rounds
                                (4096, 4096, 4096, mpg.TF32, True),          # tf32: 128 k-blocks of 32
                                (4096, 4096, 4064, mpg.TF32, False),
                                (2048, 2048, 8192, mpg.BF16_F32ACC, False)): # 64 tiles: no full round
        r = room(m, n, k, mode)
        assert ws(m, n, k, mode) == (_align256(r) + q if tail else r), (m, n, k, mode)
        assert ws(m, n, k, mode, tail_split=-1) == r
    # forced: up to SMs / 2 tiles, at any size
    assert ws(8192, 8192, 8192, mpg.BF16_F32ACC, tail_split=1) == \
        _align256(room(8192, 8192, 8192, mpg.BF16_F32ACC)) + _tail_bytes(SMS // 2)
    assert ws(512, 512, 256, mpg.BF16_F32ACC, tail_split=1) > 0
    # single-CTA tiles only (cta_pair = -1); a mode that never takes pairs
    assert ws(2560, 2560, 8192, mpg.BF16_F32ACC, cta_pair=-1) == room(2560, 2560, 8192, mpg.BF16_F32ACC)
    assert ws(2560, 2560, 8192, mpg.SPLIT_FP16_1CHAIN, prepass=-1) == 0
    # the tail follows the other regions: the conversion pass's copies first
    with_pass = ws(2560, 2560, 8192, mpg.FP16_F32ACC, prepass=1)
    pass_only = ws(2560, 2560, 8192, mpg.FP16_F32ACC, prepass=1, tail_split=-1)
    assert pass_only >= 2 * 2 * 2560 * 8192
    assert with_pass == _align256(pass_only) + q


def test_workspace_size_for_skinny_long_k(L):
    # 2048 x 128 output over k = 32768 has 16 tiles: split-K wants partials
    ws = mpg.workspace_size(2048, 128, 32768, 1, mpg.SPLIT_FP16_3CHAIN)
    assert ws > 0 and ws % (2048 * 128 * 4) == 0
    ws2 = mpg.workspace_size(2048, 128, 32768, 1, mpg.SPLIT_FP16_3CHAIN, mpg.options(splitk=4))
    assert ws2 == 4 * 2048 * 128 * 4


# ---------------------------------------------------------------- acc decode
def test_acc_coords_matches_oracle_row_col_formula(L, orc):
    for lane in range(32):
        for j in range(4):
            assert mpg.acc_coords(lane, j) == orc.acc_coords(lane, j)


def test_acc_bijection_ownership_map(L):
    seen = {}
    for lane in range(32):
        for j in range(4):
            rc = mpg.acc_coords(lane, j)
            assert rc not in seen, "overlap"
            seen[rc] = (lane, j)
    assert len(seen) == 128 and set(seen) == {(r, c) for r in range(16) for c in range(8)}


def test_acc_numeral_equals_row_col(L):
    for lane in range(32):
        for j in range(4):
            r, c = mpg.acc_coords(lane, j)
            assert mpg.acc_offset(lane, j) == r * 8 + c


def test_acc_decode_is_inverse_over_all_points(L):
    for off in range(128):
        lane, j = mpg.acc_decode(off)
        assert mpg.acc_offset(lane, j) == off
    for lane in range(32):
        for j in range(4):
            assert mpg.acc_decode(mpg.acc_offset(lane, j)) == (lane, j)
    assert mpg.acc_decode(-1) is None and mpg.acc_decode(128) is None


def test_fragment_index_split_over_two_digits(L):
    for lane in range(32):
        r0, c0 = mpg.acc_coords(lane, 0)
        assert mpg.acc_coords(lane, 1) == (r0, c0 + 1)
        assert mpg.acc_coords(lane, 2) == (r0 + 8, c0)
        assert mpg.acc_coords(lane, 3) == (r0 + 8, c0 + 1)


def test_strided_placement_stays_disjoint(L):
    # four tiles of a 32 x 24 destination with row stride 40: every offset is
    # hit by at most one (tile, lane, j) and equals (row)*stride + col
    stride, seen = 40, set()
    for tr, tc in ((0, 0), (0, 8), (16, 0), (16, 16)):
        for lane in range(32):
            for j in range(4):
                off = mpg.acc_matrix_offset(lane, j, tr, tc, stride, 32 * stride)
                r, c = mpg.acc_coords(lane, j)
                assert off == (tr + r) * stride + tc + c
                assert off not in seen
                seen.add(off)
    assert len(seen) == 4 * 128


def test_matrix_offset_overflow_and_bounds_rejected(L):
    assert mpg.acc_matrix_offset(0, 0, 0, 0, 8, 128) == 0
    assert mpg.acc_matrix_offset(31, 3, 0, 0, 8, 128) == 127
    assert mpg.acc_matrix_offset(31, 3, 0, 0, 8, 127) is None       # reaches the limit
    assert mpg.acc_matrix_offset(0, 1, 0, 7, 8, 10 ** 6) is None     # column spills past the row
    assert mpg.acc_matrix_offset(0, 0, 2 ** 62, 0, 4, 2 ** 63 - 1) is None  # int64 overflow
    assert mpg.acc_matrix_offset(0, 0, -1, 0, 8, 128) is None
    assert mpg.acc_matrix_offset(32, 0, 0, 0, 8, 128) is None
    assert mpg.acc_matrix_offset(0, 4, 0, 0, 8, 128) is None


def test_tmem_accumulator_map(L):
    rows = set()
    for warp in range(2, 6):
        for lane in range(32):
            r, c = mpg.tmem_acc_coords(warp, lane, 5, 64)
            assert c == 69
            rows.add(r)
    assert rows == set(range(128))
    assert mpg.tmem_acc_coords(0, 32, 0) is None
    assert mpg.tmem_acc_coords(0, 0, 0, 512) is None


@pytest.mark.parametrize("m_shape", [128, 256])
def test_tmem_accumulator_map_round_trips_over_every_point(L, m_shape):
    """Every (cta, warp, lane, register, load) of an m_shape x 256 accumulator
    read in 32-column loads lands on a distinct point, the points cover the
    whole accumulator (no gap, no overlap for warps 0-3; warps 4-7 repeat
    them), and the decode is the inverse, for every load width."""
    ncol = 256
    hits = {}
    for cta in range(m_shape // 128):
        for warp in range(8):
            for lane in range(32):
                for col in range(ncol):
                    cb, reg = col - col % 32, col % 32
                    r, c = mpg.tmem_acc_coords(warp, lane, reg, cb, m_shape=m_shape, cta_rank=cta)
                    hits.setdefault((r, c), []).append((cta, warp, lane, reg, cb))
    assert set(hits) == {(r, c) for r in range(m_shape) for c in range(ncol)}
    assert all(len(v) == 2 for v in hits.values())
    for (r, c), owners in hits.items():
        cta, warp, lane, reg, cb = owners[0]
        assert warp < 4 and owners[1][1] == warp + 4      # the same lanes, one warpgroup apart
        assert mpg.tmem_acc_decode(r, c, 32, m_shape=m_shape) == (cta, warp, lane, reg, cb)
    for w in (1, 2, 4, 8, 16, 64, 128):
        for r, c in ((0, 0), (m_shape - 1, 511), (77, 300), (m_shape // 2 + 5, 129)):
            cta, warp, lane, reg, cb = mpg.tmem_acc_decode(r, c, w, m_shape=m_shape)
            assert cb % w == 0 and reg < w
            assert mpg.tmem_acc_coords(warp, lane, reg, cb, m_shape=m_shape, cta_rank=cta) == (r, c)


def test_tmem_accumulator_map_rejects_bad_arguments(L):
    assert mpg.tmem_acc_coords(0, 0, 0, 0, m_shape=64) is None          # only M = 128 and M = 256
    assert mpg.tmem_acc_coords(0, 0, 0, 0, m_shape=128, cta_rank=1) is None
    assert mpg.tmem_acc_coords(0, 0, 0, 0, m_shape=256, cta_rank=2) is None
    assert mpg.tmem_acc_coords(-1, 0, 0, 0) is None
    assert mpg.tmem_acc_coords(0, 0, 511, 1) is None                     # past the 512 TMEM columns
    assert mpg.tmem_acc_decode(128, 0) is None                           # row beyond M
    assert mpg.tmem_acc_decode(0, 512) is None
    assert mpg.tmem_acc_decode(0, 0, 3) is None                          # load width not a power of two
    assert mpg.tmem_acc_decode(0, 0, 256) is None
    assert mpg.tmem_acc_decode(255, 0, m_shape=256) == (1, 3, 31, 0, 0)


# ---------------------------------------------------------------- operand fragments
def test_fragment_maps_match_oracle_definition(L, orc):
    for lane in range(32):
        for i in range(8):
            assert mpg.frag_a_coords(lane, i) == orc.frag_a_coords(lane, i)
        for i in range(4):
            assert mpg.frag_b_coords(lane, i) == orc.frag_b_coords(lane, i)


def test_fragment_maps_are_bijections_with_inverse(L):
    seen_a, seen_b = set(), set()
    for lane in range(32):
        for i in range(8):
            r, c = mpg.frag_a_coords(lane, i)
            assert 0 <= r < 16 and 0 <= c < 16 and (r, c) not in seen_a
            seen_a.add((r, c))
            assert mpg.frag_a_decode(r, c) == (lane, i)
        for i in range(4):
            k, n = mpg.frag_b_coords(lane, i)
            assert 0 <= k < 16 and 0 <= n < 8 and (k, n) not in seen_b
            seen_b.add((k, n))
            assert mpg.frag_b_decode(k, n) == (lane, i)
    assert len(seen_a) == 256 and len(seen_b) == 128
    assert mpg.frag_a_coords(32, 0) is None and mpg.frag_a_coords(0, 8) is None
    assert mpg.frag_b_coords(0, 4) is None and mpg.frag_b_decode(16, 0) is None


def test_fragment_numerals(L):
    # A: offset = (i&1) + tig*2 + (i>>2)*8 + group*16 + ((i>>1)&1)*128 (row-major)
    # B: offset = (i&1) + tig*2 + (i>>1)*8 + group*16 (column-major)
    for lane in range(32):
        g, t = lane // 4, lane % 4
        for i in range(8):
            r, c = mpg.frag_a_coords(lane, i)
            assert r * 16 + c == (i & 1) + t * 2 + (i >> 2) * 8 + g * 16 + ((i >> 1) & 1) * 128
        for i in range(4):
            k, n = mpg.frag_b_coords(lane, i)
            assert n * 16 + k == (i & 1) + t * 2 + (i >> 1) * 8 + g * 16


def test_attention_arguments_rejected_before_launch(L):
    def call(**kw):
        a = dict(lq=256, lk=512, d=128, Q=16, ldq=128, K=16, ldk=128, V=16, ldv=128, O=16, ldo=128, scale=0.1,
                 mode=mpg.ATTN_SPLIT_2CHAIN, key_splits=0)
        a.update(kw)
        return mpg.attention_raw(a["lq"], a["lk"], a["d"], a["Q"], a["ldq"], a["K"], a["ldk"], a["V"], a["ldv"],
                                 a["O"], a["ldo"], a["scale"], a["mode"], a["key_splits"], check=False)
    assert call(d=64) == mpg.ERR_UNSUPPORTED
    assert call(mode=2) == mpg.ERR_UNSUPPORTED
    assert call(lk=0) == mpg.ERR_INVALID_ARG
    assert call(ldk=120) == mpg.ERR_INVALID_ARG
    assert call(ldk=132) == mpg.ERR_INVALID_ARG          # not a multiple of 8: TMA rows
    assert call(K=24) == mpg.ERR_INVALID_ARG             # not 16-byte aligned
    assert call(Q=0) == mpg.ERR_INVALID_ARG
    assert call(key_splits=-1) == mpg.ERR_INVALID_ARG
    assert call(scale=float("inf")) == mpg.ERR_INVALID_ARG
    assert call(lq=0) == mpg.OK                          # nothing to do


def test_attention_workspace_holds_the_partials(L):
    # forced key ranges: partial outputs (128 floats per row) plus a maximum and
    # a sum per row for every range
    ws = mpg.attention_workspace_size(2048, 32768, 128, 8)
    assert ws >= 8 * 2048 * (128 + 2) * 4
    assert mpg.attention_workspace_size(2048, 32768, 128, 1) == 0
    assert mpg.attention_workspace_size(2048, 32768, 64, 0) == 0


def test_attention_key_ranges_are_at_most_one_per_block(L):
    # 1000 keys are 8 blocks of 128: asking for 8, 9 or 50 ranges gives 8, each
    # holding partial outputs (128 floats per query) plus a maximum and a sum
    # per query, every array padded to 256 bytes
    def a256(x):
        return (x + 255) // 256 * 256
    want = a256(8 * 200 * 128 * 4) + 2 * a256(8 * 200 * 4)
    for splits in (8, 9, 50):
        assert mpg.attention_workspace_size(200, 1000, 128, splits) == want
    # 1024 keys: 8 ranges of one block; 1025 keys are 9 blocks, and 8 ranges of
    # equal length would need 2 blocks each, which leaves 5 ranges (2, 2, 2, 2, 1)
    assert mpg.attention_workspace_size(200, 1024, 128, 8) == want
    assert mpg.attention_workspace_size(200, 1025, 128, 8) == a256(5 * 200 * 128 * 4) + 2 * a256(5 * 200 * 4)


def test_workspace_includes_the_conversion_pass_when_the_library_takes_it(L):
    # split modes with both operands re-read by many tiles: the library's
    # choice is the separate pass, so the query includes the hi/lo copies
    # (4 bytes per element of A and of B); never (-1) or a skinny / small
    # problem: no copies
    n = 4096
    ws = mpg.workspace_size(n, n, n, 1, mpg.SPLIT_FP16_3CHAIN)
    assert ws >= 2 * 4 * n * n
    assert mpg.workspace_size(n, n, n, 1, mpg.SPLIT_FP16_3CHAIN, mpg.options(prepass=-1)) == 0
    assert mpg.workspace_size(256, 256, 256, 1, mpg.SPLIT_FP16_3CHAIN) == 0
    never = mpg.options(tail_split=-1, prepass=-1)
    assert mpg.workspace_size(n, n, n, 1, mpg.FP16_F32ACC, never) == 0   # fp16 mode, pass refused
    assert mpg.workspace_size(n, n, n, 1, mpg.FP16_F32ACC, mpg.options(prepass=1)) >= 2 * 2 * n * n
    assert _call(opts=mpg.options(prepass=2)) == mpg.ERR_INVALID_ARG


def test_exact_query_includes_the_pass_for_fp16_modes_on_fp32_operands(L):
    n = 4096
    nt = mpg.options(tail_split=-1)     # without the split tail's partial sums
    plain = mpg.workspace_size(n, n, n, 1, mpg.FP16_F32ACC, nt)
    exact = mpg.workspace_size_ex(n, n, n, 1, 256, n, 0, mpg.F32, mpg.ROW_MAJOR, 256, n, 0, mpg.F32,
                                  mpg.ROW_MAJOR, mpg.FP16_F32ACC, nt)
    assert exact >= 2 * 2 * n * n and plain >= exact        # fp16 copies of A and B
    exact16 = mpg.workspace_size_ex(n, n, n, 1, 256, n, 0, mpg.F16, mpg.ROW_MAJOR, 256, n, 0, mpg.F16,
                                    mpg.ROW_MAJOR, mpg.FP16_F32ACC, nt)
    assert exact16 == 0                                      # fp16 operands: nothing to convert
    never = mpg.workspace_size_ex(n, n, n, 1, 256, n, 0, mpg.F32, mpg.ROW_MAJOR, 256, n, 0, mpg.F32,
                                  mpg.ROW_MAJOR, mpg.FP16_F32ACC, mpg.options(prepass=-1, tail_split=-1))
    assert never == 0
    # with the split tail (k >= 8192): it follows the copies
    k = 8192
    copies = mpg.workspace_size_ex(n, n, k, 1, 256, k, 0, mpg.F32, mpg.ROW_MAJOR, 256, n, 0, mpg.F32,
                                   mpg.ROW_MAJOR, mpg.FP16_F32ACC, nt)
    full = mpg.workspace_size_ex(n, n, k, 1, 256, k, 0, mpg.F32, mpg.ROW_MAJOR, 256, n, 0, mpg.F32,
                                 mpg.ROW_MAJOR, mpg.FP16_F32ACC)
    assert copies >= 2 * (n * k + k * n) and full == _align256(copies) + _tail_bytes(SMS // 4)
